// attn_tc.cu -- non-causal block attention over the paged KV cache on the
// 5th-generation tensor cores.
//
// One CTA per work item (sequence, kv head, split of the keys [cached context
// ; 16 block rows]).  The G q-heads x 16 block rows that share a kv head form
// one M = 128 query tile (rows padded with zeros when G*16 < 128), so each
// K/V page is read once per item.  Keys go in chunks of two pages (128 keys):
// one S tile per chunk halves the serial S -> softmax -> P V^T steps of a
// split.
//   warp 0 (one lane)  TMA: the query tile, then the split's K pages [64 x d]
//                      and V^T pages [d x 64] into a ring of chunk stages
//                      (three at d = 128; a chunk's two K pages stacked to
//                      one 128-key operand);
//   warp 1 (one lane)  tcgen05.mma: S = Q K^T (N = 128) into one of two TMEM
//                      buffers, then O += P V^T into the TMEM accumulator
//                      with P read from TMEM, issued in dependency order;
//   warps 2..9         softmax, two threads per query row (warps 2..5 the
//                      chunk's first 64 keys, warps 6..9 the other 64; the
//                      two halves trade their maxima through TMEM): scores
//                      from TMEM, exp2 with a running max, P (bf16 pairs)
//                      written back over the half's own scores, so chunk
//                      c+1's softmax overlaps chunk c's P V^T and shared
//                      memory holds only Q and the K/V ring.  O is rescaled
//                      only when a row's max grows by more than 2^8 (exact:
//                      the final division uses the same max); each half
//                      rescales half of O's columns.
// Each item writes its unnormalised O with (max, sum); the combine kernel
// merges the splits (all in log2 units).
#include <algorithm>
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

struct AttnTcCfg {
  int datoms;        // d / 64 (K-atoms of a row)
  int stages;        // chunk stages
  int stage_bytes;   // datoms x 16 KB of K (two pages stacked) + 2 x V^T page (d x 128 B)
  uint32_t idesc_s;  // M=128, N=128
  uint32_t idesc_o;  // M=128, N=d
  float scale_log2;  // log2(e) / sqrt(d)
};

constexpr int kAttnThreads = 320;
constexpr int kSmThreads = 256;          // softmax warps 2..9
constexpr int kSmBar = 3;                // their named barrier
constexpr int kQAtomBytes = 128 * 128;   // 128 rows x 128 B
constexpr int kKAtomBytes = 64 * 128;    // 64 keys x 128 B (one page of one K-atom)
constexpr int kChunk = 2 * kPage;        // keys per S tile
constexpr int kMaxAttnStages = 4;
constexpr float kRescaleLog2 = 8.f;

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, AttnArgs a, AttnTcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geo& g = a.g;
  uint8_t* sQ = smem;                                   // datoms x 16 KB
  uint8_t* sKV = sQ + t.datoms * kQAtomBytes;           // stages x stage_bytes
  uint8_t* ctl = sKV + t.stages * t.stage_bytes;
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
  const uint32_t vbytes = (uint32_t)g.d * 128;          // one V^T page
  // zero the query tile's padding rows (the MMA reads all 128 rows)
  for (int idx = threadIdx.x; idx < t.datoms * (128 - R) * 32; idx += kAttnThreads) {
    const int atom = idx / ((128 - R) * 32), rem = idx % ((128 - R) * 32);
    reinterpret_cast<uint32_t*>(sQ + atom * kQAtomBytes + R * 128)[rem] = 0u;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(qfull, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], kSmThreads);
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

  // The descriptor, the page table and the cached-context pages were written
  // by kernels that completed before the predecessor passed its own launch
  // wait (which is when this kernel may start), so they are read before this
  // kernel's wait; only the pages holding this round's block rows and the
  // query tile (both written by the predecessor) wait for it.
  const int item = a.rd->perm[blockIdx.x];              // longest items launch first
  int s, kvh, k0, k1, ks;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1, &ks);
  const int n_pages = (k1 - k0 + kPage - 1) / kPage;
  const int n_chunks = (n_pages + 1) / 2;
  const int slot = a.rd->seq_slot[s];
  const int len = a.rd->len[s];
  auto pages_in = [&](int c) { return min(2, n_pages - 2 * c); };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      // page j of the split goes to chunk stage (j/2) % stages, K rows
      // [64*(j&1), +64) of each K-atom and V^T slot j&1
      auto load_page = [&](int j) -> bool {
        const int st = (j >> 1) % t.stages, w = j & 1;
        const int page = a.block_table[(long)slot * g.pages_per_seq + k0 / kPage + j];
        if (page < 0 || page >= g.max_pages) {
          atomicExch(a.err, DERR_BAD_PAGE);
          return false;
        }
        const long base = ((long)a.layer * g.max_pages + page) * g.Hkv + kvh;
        uint8_t* st_k = sKV + st * t.stage_bytes;
        uint8_t* st_v = st_k + t.datoms * kQAtomBytes;
        for (int at = 0; at < t.datoms; ++at)
          tma_load_2d(st_k + at * kQAtomBytes + w * kKAtomBytes, &tmK, &kvfull[st], at * 64, (int)(base * kPage));
        tma_load_2d(st_v + w * vbytes, &tmV, &kvfull[st], 0, (int)(base * g.d));
        return true;
      };
      auto chunk_bytes = [&](int c) { return (uint32_t)(pages_in(c) * (t.datoms * kKAtomBytes + (int)vbytes)); };
      bool ok = true;
      int deferred[2 * kMaxAttnStages];
      int nd = 0;
      // the first chunk stage is free: announce it and fetch its
      // context-only pages before the launch wait (one stage only: the
      // query tile, loaded after the wait, queues behind what is in flight)
      const int pre = min(n_chunks, 1);
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
      mbar_arrive_expect_tx(qfull, (uint32_t)(t.datoms * R * 128));
      for (int at = 0; at < t.datoms; ++at)
        tma_load_3d(sQ + at * kQAtomBytes, &tmQ, qfull, at * 64, kvh * g.G, s * kBlock);
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
      const uint32_t q_addr = smem_u32(sQ);
      auto kv_addr = [&](int c) -> uint32_t { return smem_u32(sKV + (c % t.stages) * t.stage_bytes); };
      // S(c) = Q K(c)^T, once the caller has seen chunk c's keys land
      auto issue_s = [&](int c) {
        tc_fence_after();
        const uint32_t k_addr = kv_addr(c);
        const uint32_t d_s = tmem + 128u + (uint32_t)((c & 1) * kChunk);
        for (int kk = 0; kk < 4 * t.datoms; ++kk) {
          const int at = kk >> 2;
          const uint64_t adv = (uint64_t)((kk & 3) * 32) >> 4;
          mma_bf16(d_s, desc_sw128(q_addr + at * kQAtomBytes) + adv, desc_sw128(k_addr + at * kQAtomBytes) + adv,
                   t.idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sfull[c & 1]);
      };
      // O += P(c) V(c)^T, once the caller has seen softmax(c) publish P.
      // P of key half h sits in columns [64h, 64h + 32) of S buffer c&1
      // (two keys per column), so a 16-key step reads 8 columns.
      auto issue_pv = [&](int c) {
        tc_fence_after();
        const uint32_t p_tmem = tmem + 128u + (uint32_t)((c & 1) * kChunk);
        const uint32_t v_addr = kv_addr(c) + (uint32_t)(t.datoms * kQAtomBytes);
        const int steps = pages_in(c) * (kPage / 16);   // 16 keys per MMA; a missing second page is skipped
        for (int kk = 0; kk < steps; ++kk) {
          const int pa = kk >> 2;                        // page (key half / V^T slot) of this K-step
          const uint64_t adv = (uint64_t)((kk & 3) * 32) >> 4;
          mma_f16_ts(tmem, p_tmem + (uint32_t)(pa * kPage + (kk & 3) * 8), desc_sw128(v_addr + pa * vbytes) + adv,
                      t.idesc_o, (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pvdone[c & 1]);
        mma_commit(&kvempty[c % t.stages]);
      };
      // Issue in dependency order rather than program order: S(ns) once its
      // keys have landed and S buffer ns&1 is free (softmax(ns-2) is done
      // with it and PV(ns-2), which reads P from it, was issued before: the
      // tensor pipe runs one thread's MMAs in issue order); PV(np) once
      // softmax(np) has written P.  Polling both keeps a K/V refill still in
      // flight from holding back the P V^T of the chunk before it, whose
      // completion frees the next stage.
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
    // ------------------------------------------------------------------ softmax warps
    pdl_wait();
    const int q = warp & 3;
    const int hg = (warp - 2) >> 2;              // key half of every chunk (and half of O's columns)
    const int r = 32 * q + lane;                 // query row of this thread
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t xcol = tmem + lane_base + 384u;   // exchange columns: [c&1][half] maxima, then [half] sums
    const int ocols = g.d / 2;                   // O columns this half rescales / writes
    float m_run = -INFINITY, l_run = 0.f;        // l_run: this half's share of the row sum
    bool ok = true;
    auto sm_sync = [&]() { asm volatile("barrier.sync %0, %1;" ::"r"(kSmBar), "r"(kSmThreads) : "memory"); };
    for (int c = 0; c < n_chunks; ++c) {
      // a failed wait still reaches every barrier below (skipping the work)
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sfull[c & 1], (c >> 1) & 1, &flags[0]));
      if (!got) ok = false;
      __syncwarp();
      tc_fence_after();
      float sc[kPage];
      const uint32_t sbase = tmem + lane_base + 128u + (uint32_t)((c & 1) * kChunk + hg * kPage);
      const int kbase = k0 + c * kChunk + hg * kPage;
      const int kc = min(kPage, k1 - kbase);   // valid keys of this half (may be <= 0)
      const int klo = ks - kbase;              // keys below the window start (first page only)
      // raw scores (masked keys -inf; whole pages skip the mask); the
      // log2-domain scale is applied to the maximum and inside exp2's argument
      float mh = -INFINITY;
      if (ok) {
        tmem_ld32(sbase, sc);
        tmem_ld32(sbase + 32u, sc + 32);
        if (kc >= kPage && klo <= 0) {
#pragma unroll
          for (int i = 0; i < kPage; ++i) mh = fmaxf(mh, sc[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kPage; ++i) {
            sc[i] = (i < kc && i >= klo) ? sc[i] : -INFINITY;
            mh = fmaxf(mh, sc[i]);
          }
        }
      }
      tmem_st1(xcol + (uint32_t)(2 * (c & 1) + hg), mh);
      tc_fence_before();
      sm_sync();
      tc_fence_after();
      const float mj = t.scale_log2 * fmaxf(mh, tmem_ld1(xcol + (uint32_t)(2 * (c & 1) + (hg ^ 1))));
      if (!ok || flags[0]) {
        ok = false;
        mbar_arrive(&pfull[c & 1]);
        continue;
      }
      const bool need = mj > m_run + kRescaleLog2;
      const bool resc = __any_sync(0xffffffffu, need && c > 0);
      // rescaling O needs every product issued so far (through chunk c-1) done
      if (resc) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pvdone[(c - 1) & 1], ((c - 1) >> 1) & 1, &flags[0]))) {
          ok = false;
          mbar_arrive(&pfull[c & 1]);
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
      float lsum = 0.f;
      // P over this half's own scores (both halves loaded theirs before the
      // max exchange): 32 columns of bf16 pairs
      const float nm = -m_run;
      float pw[kPage / 2];
#pragma unroll
      for (int i = 0; i < kPage / 2; ++i) {
        const float p0 = ex2_fast(fmaf(sc[2 * i], t.scale_log2, nm));
        const float p1 = ex2_fast(fmaf(sc[2 * i + 1], t.scale_log2, nm));
        lsum += p0 + p1;
        const __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);
        pw[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&b));
      }
      tmem_st32(sbase, pw);
      l_run += lsum;
      tc_fence_before();
      mbar_arrive(&pfull[c & 1]);
    }
    bool fin = ok && n_chunks > 0 &&
               __all_sync(0xffffffffu, mbar_wait(&pvdone[(n_chunks - 1) & 1], ((n_chunks - 1) >> 1) & 1, &flags[0]));
    __syncwarp();
    tc_fence_after();
    // the row sum is the two halves' shares
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
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow * g.d + hg * ocols + cc * 32);
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
  __syncwarp();   // role lanes rejoin their warp before the CTA barrier
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 5, c0);     // 5: exit
  if (threadIdx.x == 64) trace_mark(a.trace, blockIdx.x, 7, c0);
  trace_exit_warp(a.trace, blockIdx.x);
  if (flags[0] && threadIdx.x == 0) atomicExch(a.err, DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t attn_tc_smem_bytes(int d, int stages) {
  const int datoms = d / 64;
  const int stage_bytes = datoms * kQAtomBytes + 2 * d * 128;
  return (size_t)datoms * kQAtomBytes + (size_t)stages * stage_bytes + 256 + 1024;
}

// As many chunk stages as 227 KB of shared memory holds (at most four).
static int attn_tc_stages(int d) {
  int st = kMaxAttnStages;
  while (st > 2 && attn_tc_smem_bytes(d, st) > 227u * 1024u) --st;
  return st;
}

void launch_attention_tc(const AttnArgs& a, int n_items, const void* tmq, const void* tmk, const void* tmv,
                         cudaStream_t s) {
  AttnTcCfg t{};
  const int d = a.g.d;
  t.datoms = d / 64;
  t.stage_bytes = t.datoms * kQAtomBytes + 2 * d * 128;
  t.stages = attn_tc_stages(d);
  t.idesc_s = idesc_bf16(128, kChunk);
  t.idesc_o = idesc_bf16(128, d);
  t.scale_log2 = 1.4426950408889634f / std::sqrt((float)d);
  const size_t smem = attn_tc_smem_bytes(d, t.stages);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;
    attr_bytes = smem;
  }
  launch_pdl(attn_tc_kernel, dim3(n_items), dim3(kAttnThreads), smem, s, *static_cast<const CUtensorMap*>(tmq),
             *static_cast<const CUtensorMap*>(tmk), *static_cast<const CUtensorMap*>(tmv), a, t);
}

}  // namespace dfl
