// attn_tc8.cu -- non-causal block attention over an e4m3 paged KV cache.
//
// The cache keeps K and V as OCP e4m3 codes with one f32 scale per (layer,
// page row, kv head); the queries arrive the same way, one scale per
// (token, q head).  Work items are those of attn_tc.cu (sequence, kv head,
// split of [cached context ; 16 block rows], the G x 16 query rows of a kv
// head as one M = 128 tile), keys in chunks of two pages:
//   warp 0 (one lane)  TMA: the e4m3 query tile [128 x 128 B], then per page
//                      K codes [64 keys x 128 B] (128-byte swizzle, the
//                      score MMA's B operand as stored), V^T codes [d x 64 B]
//                      and the page's K and V scales into a ring of chunk
//                      stages (33 KB each, four);
//   warp 1 (one lane)  tcgen05.mma: S = Q K^T with kind::f8f6f4 (both
//                      operands e4m3, straight from the ring) into one of two
//                      TMEM buffers; O += P V^T with kind::f16 (P f16 from
//                      TMEM, V f16 from shared memory); issued in dependency
//                      order as in attn_tc.cu;
//   warps 2..9         per chunk: V^T codes times their row scales -> f16
//                      into one of two shared buffers in the 128-byte
//                      swizzle, then the softmax of attn_tc.cu (two threads
//                      per query row) on scores times K scale times q scale
//                      (the latter folded into the exp2 argument), P (f16)
//                      written back over the scores.  The ring stage is
//                      released once its V is converted and its scores read.
#include <algorithm>
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

struct AttnTc8Cfg {
  int stages;
  uint32_t idesc_s;   // kind::f8f6f4 e4m3 x e4m3, M = 128, N = 128
  uint32_t idesc_o;   // kind::f16 f16 x f16, M = 128, N = d
  float scale_log2;   // log2(e) / sqrt(d)
};

constexpr int kA8Threads = 320;
constexpr int kA8SmThreads = 256;           // warps 2..9
constexpr int kA8SmBar = 3;
constexpr int kA8D = 128;                   // head dim (one 128-byte e4m3 row)
constexpr int kA8QBytes = 128 * kA8D;       // query tile
constexpr int kA8KPage = kPage * kA8D;      // 8 KB of K codes per page
constexpr int kA8VPage = kA8D * kPage;      // 8 KB of V^T codes per page
constexpr int kA8Stage = 2 * kA8KPage + 2 * kA8VPage + 4 * kPage * 4;   // + K and V scales of two pages
constexpr int kA8V16Page = kA8D * 128;      // f16 V^T page: d rows x 64 keys x 2 B
constexpr int kA8V16 = 2 * kA8V16Page;      // one chunk
constexpr int kA8MaxStages = 4;
constexpr int kA8Chunk = 2 * kPage;
constexpr float kA8RescaleLog2 = 8.f;

__global__ void __launch_bounds__(kA8Threads, 1)
    attn_tc8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, AttnArgs a, AttnTc8Cfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geo& g = a.g;
  uint8_t* sQ = smem;                                   // 16 KB
  uint8_t* sV16 = sQ + kA8QBytes;                       // 2 x 32 KB
  uint8_t* sKV = sV16 + 2 * kA8V16;                     // stages x 33 KB
  uint8_t* ctl = sKV + t.stages * kA8Stage;
  uint64_t* kvfull = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* kvempty = kvfull + t.stages;
  uint64_t* sfull = kvempty + t.stages;                 // [2]
  uint64_t* qfull = sfull + 2;
  uint64_t* pfull = qfull + 1;                          // [2]
  uint64_t* pvdone = pfull + 2;                         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pvdone + 2);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long c0 = 0;
  if (threadIdx.x == 0) trace_entry(a.trace, blockIdx.x, &c0);
  if (a.trace) {
    __shared__ unsigned long long c0_shared;
    if (threadIdx.x == 0) c0_shared = c0;
    __syncthreads();
    c0 = c0_shared;
  }
  const int R = g.G * kBlock;
  // zero the query tile's padding rows (the MMA reads all 128 rows)
  for (int idx = threadIdx.x; idx < (128 - R) * 32; idx += kA8Threads)
    reinterpret_cast<uint32_t*>(sQ + R * 128)[idx] = 0u;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], kA8SmThreads);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(qfull, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], kA8SmThreads);
      mbar_init(&pvdone[b], 1);
    }
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;                     // O: cols [0, d); S / P buffers at 128 and 256
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 1, c0);  // 1: set-up done

  const int item = blockIdx.x;
  int s, kvh, k0, k1, ks;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1, &ks);
  const int n_pages = (k1 - k0 + kPage - 1) / kPage;
  const int n_chunks = (n_pages + 1) / 2;
  const int slot = a.rd->seq_slot[s];
  const int len = a.rd->len[s];
  auto pages_in = [&](int c) { return min(2, n_pages - 2 * c); };
  auto stage_of = [&](int c) { return sKV + (c % t.stages) * kA8Stage; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      const uint64_t pol = policy_evict_first();
      const float* ksc = fp8_pool_scales(g, a.kpool);
      const float* vsc = fp8_pool_scales(g, a.vpool);
      // page j of the split: K codes at stage + (j&1) x 8 KB (the chunk's two
      // pages stack to one 128-key operand), V^T codes after both, then the
      // K scales [2][64] and V scales [2][64]
      auto load_page = [&](int j) -> bool {
        const int w = j & 1;
        const int page = a.block_table[(long)slot * g.pages_per_seq + k0 / kPage + j];
        if (page < 0 || page >= g.max_pages) {
          atomicExch(a.err, DERR_BAD_PAGE);
          return false;
        }
        const long base = ((long)a.layer * g.max_pages + page) * g.Hkv + kvh;
        uint8_t* st = stage_of(j >> 1);
        uint64_t* bar = &kvfull[(j >> 1) % t.stages];
        tma_load_2d(st + w * kA8KPage, &tmK, bar, 0, (int)(base * kPage));
        tma_load_2d(st + 2 * kA8KPage + w * kA8VPage, &tmV, bar, 0, (int)(base * kA8D));
        float* sc = reinterpret_cast<float*>(st + 2 * kA8KPage + 2 * kA8VPage);
        bulk_load_hint(sc + w * kPage, ksc + base * kPage, kPage * 4, bar, pol);
        bulk_load_hint(sc + (2 + w) * kPage, vsc + base * kPage, kPage * 4, bar, pol);
        return true;
      };
      auto chunk_bytes = [&](int c) { return (uint32_t)(pages_in(c) * (kA8KPage + kA8VPage + 2 * kPage * 4)); };
      bool ok = true;
      int deferred[2 * kA8MaxStages];
      int nd = 0;
      // the first chunk stages are free: announce them and fetch their
      // context-only pages before the launch wait (the pages holding this
      // round's block rows are written by the predecessor)
      const int pre = min(n_chunks, t.stages);
      for (int c = 0; c < pre; ++c) {
        mbar_arrive_expect_tx(&kvfull[c], chunk_bytes(c));
        for (int w = 0; w < pages_in(c); ++w) {
          const int j = 2 * c + w;
          if (k0 + (j + 1) * kPage <= len) ok = ok && load_page(j);
          else deferred[nd++] = j;
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      mbar_arrive_expect_tx(qfull, (uint32_t)(R * 128));
      tma_load_3d(sQ, &tmQ, qfull, 0, kvh * g.G, s * kBlock);
      for (int i = 0; i < nd && ok; ++i) ok = load_page(deferred[i]);
      for (int c = pre; c < n_chunks && ok; ++c) {
        const int st = c % t.stages;
        if (!mbar_wait(&kvempty[st], ((c / t.stages) & 1) ^ 1, &flags[0])) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kvfull[st], chunk_bytes(c));
        for (int w = 0; w < pages_in(c) && ok; ++w) ok = load_page(2 * c + w);
      }
      if (!ok) flags[0] = 1;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(qfull, 0, &flags[0]);
      tc_fence_after();
      trace_mark(a.trace, blockIdx.x, 2, c0);                   // 2: query tile ready
      const uint64_t dq = desc_sw128(smem_u32(sQ));
      // S(c) = Q K(c)^T: e4m3 rows of 128 bytes, 32 per instruction
      auto issue_s = [&](int c) {
        tc_fence_after();
        const uint64_t dk = desc_sw128(smem_u32(stage_of(c)));
        const uint32_t d_s = tmem + 128u + (uint32_t)((c & 1) * kA8Chunk);
#pragma unroll
        for (int kk = 0; kk < kA8D / 32; ++kk) mma_f8(d_s, dq + 2 * kk, dk + 2 * kk, t.idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(&sfull[c & 1]);
      };
      // O += P'(c) V(c)^T: P' f16 in columns [64h, 64h + 32) of S buffer c&1
      // for key half h, V^T f16 page h in shared buffer c&1
      auto issue_pv = [&](int c) {
        tc_fence_after();
        const uint32_t p_tmem = tmem + 128u + (uint32_t)((c & 1) * kA8Chunk);
        const uint32_t v_addr = smem_u32(sV16 + (c & 1) * kA8V16);
        const int steps = pages_in(c) * (kPage / 16);
        for (int kk = 0; kk < steps; ++kk) {
          const int pa = kk >> 2;
          mma_f16_ts(tmem, p_tmem + (uint32_t)(pa * kPage + (kk & 3) * 8),
                     desc_sw128(v_addr + pa * kA8V16Page) + (uint64_t)(2 * (kk & 3)), t.idesc_o,
                     (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pvdone[c & 1]);
      };
      // dependency order: S(ns) once its stage landed and S buffer ns&1 is
      // free (PV(ns-2) issued); PV(np) once the softmax warps published P'
      // and the f16 V of chunk np
      int ns = 0, np = 0;
      uint64_t t_last = globaltimer();
      while (ok && np < n_chunks) {
        bool prog = false;
        if (np < ns && mbar_try_wait(&pfull[np & 1], (np >> 1) & 1)) {
          issue_pv(np++);
          prog = true;
        }
        if (ns < n_chunks && ns <= np + 1 && mbar_try_wait(&kvfull[ns % t.stages], (ns / t.stages) & 1)) {
          issue_s(ns++);
          prog = true;
        }
        if (prog) t_last = globaltimer();
        else if (flags[0] || globaltimer() - t_last > kWaitNs) ok = false;
      }
      if (!ok) flags[0] = 1;
      trace_mark(a.trace, blockIdx.x, 3, c0);                   // 3: last MMA issued
    }
  } else {
    // ------------------------------------------------------------------ convert + softmax warps
    pdl_wait();
    const int q = warp & 3;
    const int hg = (warp - 2) >> 2;              // key half of every chunk (and half of O's columns)
    const int r = 32 * q + lane;                 // query row of this thread
    const int ct = threadIdx.x - 64;             // 0..255: converter index
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t xcol = tmem + lane_base + 384u;
    const int ocols = kA8D / 2;
    // this row's query scale folded into the log2-domain score scale
    // (positive for every row, padding rows included)
    float a_row = t.scale_log2;
    if (r < R) {
      const float* qs = reinterpret_cast<const float*>(static_cast<const char*>(a.q) + fp8_q_codes(g));
      a_row *= qs[(long)(s * kBlock + r / g.G) * g.Hq + kvh * g.G + r % g.G];
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    auto sm_sync = [&]() { asm volatile("barrier.sync %0, %1;" ::"r"(kA8SmBar), "r"(kA8SmThreads) : "memory"); };
    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % t.stages;
      const uint8_t* stp = stage_of(c);
      const float* ssc = reinterpret_cast<const float*>(stp + 2 * kA8KPage + 2 * kA8VPage);
      // (1) the stage has landed and V buffer c&1 is free (PV(c-2) done)
      bool got = __all_sync(0xffffffffu, mbar_wait(&kvfull[st], (c / t.stages) & 1, &flags[0]));
      if (got && c >= 2) got = __all_sync(0xffffffffu, mbar_wait(&pvdone[c & 1], ((c - 2) >> 1) & 1, &flags[0]));
      if (!got) ok = false;
      __syncwarp();
      // (2) V^T codes x V scales -> f16: 16-key pieces, (page, d row,
      // piece) per item; a warp reads 512 contiguous bytes and writes 8 whole
      // 128-byte rows
      if (ok) {
        uint8_t* vdst = sV16 + (c & 1) * kA8V16;
        for (int it = ct; it < pages_in(c) * kA8D * 4; it += kA8SmThreads) {
          const int w = it >> 9, row = (it >> 2) & (kA8D - 1), pc = it & 3;
          const uint4 src = *reinterpret_cast<const uint4*>(stp + 2 * kA8KPage + w * kA8VPage + row * kPage + pc * 16);
          const float4* svp = reinterpret_cast<const float4*>(ssc + (2 + w) * kPage + pc * 16);
          const uint32_t sw[4] = {src.x, src.y, src.z, src.w};
          uint32_t h[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 sv4 = svp[i];   // scales of keys 4i .. 4i+3 of the piece
            const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(sw[i] & 0xFFFFu), __NV_E4M3);
            const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(sw[i] >> 16), __NV_E4M3);
            const __half2 vlo = __hmul2(__half2(lo), __floats2half2_rn(sv4.x, sv4.y));
            const __half2 vhi = __hmul2(__half2(hi), __floats2half2_rn(sv4.z, sv4.w));
            h[2 * i] = *reinterpret_cast<const uint32_t*>(&vlo);
            h[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&vhi);
          }
          uint8_t* drow = vdst + w * kA8V16Page + row * 128;
          *reinterpret_cast<uint4*>(drow + (((2 * pc) ^ (row & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(drow + (((2 * pc + 1) ^ (row & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
      fence_proxy_async_smem();
      // (3) scores
      got = __all_sync(0xffffffffu, ok && mbar_wait(&sfull[c & 1], (c >> 1) & 1, &flags[0]));
      if (!got) ok = false;
      __syncwarp();
      tc_fence_after();
      float sc[kPage];
      const uint32_t sbase = tmem + lane_base + 128u + (uint32_t)((c & 1) * kA8Chunk + hg * kPage);
      const int kbase = k0 + c * kA8Chunk + hg * kPage;
      const int kc = min(kPage, k1 - kbase);   // valid keys of this half (may be <= 0)
      const int klo = ks - kbase;              // keys below the window start (first page only)
      const float* sk = ssc + hg * kPage;      // K scales of this half's page
      // scores times K scales (masked keys -inf; whole pages skip the mask)
      float mh = -INFINITY;
      if (ok) {
        tmem_ld32(sbase, sc);
        tmem_ld32(sbase + 32u, sc + 32);
        if (kc >= kPage && klo <= 0) {
#pragma unroll
          for (int i = 0; i < kPage; ++i) {
            sc[i] *= sk[i];
            mh = fmaxf(mh, sc[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kPage; ++i) {
            sc[i] = (i < kc && i >= klo) ? sc[i] * sk[i] : -INFINITY;
            mh = fmaxf(mh, sc[i]);
          }
        }
      }
      tmem_st1(xcol + (uint32_t)(2 * (c & 1) + hg), mh);
      tc_fence_before();
      sm_sync();
      tc_fence_after();
      // the row maximum in log2 units (a_row > 0 keeps the order)
      const float mj = a_row * fmaxf(mh, tmem_ld1(xcol + (uint32_t)(2 * (c & 1) + (hg ^ 1))));
      if (!ok || flags[0]) {
        ok = false;
        mbar_arrive(&pfull[c & 1]);
        mbar_arrive(&kvempty[st]);
        continue;
      }
      const bool need = mj > m_run + kA8RescaleLog2;
      const bool resc = __any_sync(0xffffffffu, need && c > 0);
      // rescaling O needs every product issued so far (through chunk c-1) done
      if (resc) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pvdone[(c - 1) & 1], ((c - 1) >> 1) & 1, &flags[0]))) {
          ok = false;
          mbar_arrive(&pfull[c & 1]);
          mbar_arrive(&kvempty[st]);
          continue;
        }
        __syncwarp();
        tc_fence_after();
        const float alpha = need ? exp2f(m_run - mj) : 1.f;
        for (int cc = 0; cc < ocols / 32; ++cc) {
          float o[32];
          const uint32_t oa = tmem + lane_base + (uint32_t)(hg * ocols + cc * 32);
          tmem_ld32(oa, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(oa, o);
        }
        l_run *= alpha;
      }
      if (need) m_run = mj;
      // (4) P = 2^(a_row t - m) (f16 pairs) over this half's own scores;
      // masked keys (t = -inf) give exact zeros
      const float nm = -m_run;
      float lsum = 0.f;
      float pw[kPage / 2];
#pragma unroll
      for (int i = 0; i < kPage / 2; ++i) {
        const float p0 = ex2_fast(fmaf(sc[2 * i], a_row, nm));
        const float p1 = ex2_fast(fmaf(sc[2 * i + 1], a_row, nm));
        lsum += p0 + p1;
        const __half2 hp = __floats2half2_rn(p0, p1);
        pw[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&hp));
      }
      tmem_st32(sbase, pw);
      l_run += lsum;
      tc_fence_before();
      mbar_arrive(&pfull[c & 1]);
      mbar_arrive(&kvempty[st]);   // K read by S(c), V converted, scales read
    }
    bool fin = ok && n_chunks > 0 &&
               __all_sync(0xffffffffu, mbar_wait(&pvdone[(n_chunks - 1) & 1], ((n_chunks - 1) >> 1) & 1, &flags[0]));
    __syncwarp();
    tc_fence_after();
    tmem_st1(xcol + 4u + (uint32_t)hg, l_run);
    tc_fence_before();
    sm_sync();
    tc_fence_after();
    const float l_tot = l_run + tmem_ld1(xcol + 4u + (uint32_t)(hg ^ 1));
    if (fin) {
      const long prow = (long)item * R + r;
      for (int cc = 0; cc < ocols / 32; ++cc) {
        float o[32];
        tmem_ld32(tmem + lane_base + (uint32_t)(hg * ocols + cc * 32), o);
        if (r < R) {
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow * kA8D + hg * ocols + cc * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      if (r < R && hg == 0) {
        a.part_ml[prow * 2] = m_run;
        a.part_ml[prow * 2 + 1] = l_tot;
      }
    } else if (n_chunks > 0) {
      flags[0] = 1;
    }
  }
  if (threadIdx.x == 64) trace_mark(a.trace, blockIdx.x, 4, c0);   // 4: softmax warps done
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 5, c0);     // 5: exit
  if (threadIdx.x == 64) trace_mark(a.trace, blockIdx.x, 7, c0);
  if (threadIdx.x == 0) trace_exit(a.trace, blockIdx.x);
  if (flags[0] && threadIdx.x == 0) atomicExch(a.err, DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t attn_tc8_smem_bytes(int stages) {
  return (size_t)kA8QBytes + 2 * kA8V16 + (size_t)stages * kA8Stage + 256 + 1024;
}

void launch_attention_tc8(const AttnArgs& a, int n_items, const void* tmq, const void* tmk, const void* tmv,
                          cudaStream_t s) {
  if (a.g.d != kA8D) return;   // create() admits e4m3 caches only at d = 128
  AttnTc8Cfg t{};
  t.stages = kA8MaxStages;
  while (t.stages > 2 && attn_tc8_smem_bytes(t.stages) > 227u * 1024u) --t.stages;
  t.idesc_s = idesc_fmt0(128, kA8Chunk);
  t.idesc_o = idesc_fmt0(128, kA8D);
  t.scale_log2 = 1.4426950408889634f / std::sqrt((float)kA8D);
  const size_t smem = attn_tc8_smem_bytes(t.stages);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(attn_tc8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;
    attr_bytes = smem;
  }
  launch_pdl(attn_tc8_kernel, dim3(n_items), dim3(kA8Threads), smem, s, *static_cast<const CUtensorMap*>(tmq),
             *static_cast<const CUtensorMap*>(tmk), *static_cast<const CUtensorMap*>(tmv), a, t);
}

}  // namespace dfl
