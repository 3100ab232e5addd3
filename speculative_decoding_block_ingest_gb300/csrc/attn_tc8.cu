// attn_tc8.cu -- non-causal block attention over an e4m3 paged KV cache.
//
// The cache keeps K and V as OCP e4m3 codes with one f32 scale per (layer,
// page row, kv head) (spark_model::layers::dflash_head, the FP8 block
// attention kernel named in the module summary; DflashQuantization).  Only
// the storage is e4m3: the queries stay f16 and both products run on the
// kind::f16 tensor cores, so the scores are those of the cached values.
// Work items are those of attn_tc.cu (sequence, kv head, split of [cached
// context ; 16 block rows], the G x 16 query rows of a kv head as one
// M = 128 tile), keys in chunks of two pages:
//   warp 0 (one lane)  TMA: the f16 query tile, then per page the K codes
//                      [64 keys x 128 B] (128-byte swizzle), the V^T codes
//                      [d x 64 B] and the page's K and V scales into a ring
//                      of raw chunk stages (the first ones before the
//                      programmatic-launch wait);
//   warps 10, 11       converters, per chunk: K codes -> f16 times 2^-8
//                      (exact, by integer operations) into the chunk's K
//                      operand, the chunk's K scales into one of three small
//                      buffers;
//   warp 1 (one lane)  tcgen05.mma: S = Q K^T into one of two TMEM buffers,
//                      O += P V^T with P read from TMEM, issued in dependency
//                      order as in attn_tc.cu;
//   warps 2..9         per chunk, first V^T codes times their row scales (the
//                      product in f32, where it is exact, rounded once) ->
//                      f16 into one of two V operands (these warps would
//                      otherwise wait for the scores), then the softmax of
//                      attn_tc.cu (two threads per query row) on the scores
//                      times their keys' scales; P (f16) written back over
//                      the scores.
// A raw stage is free once both groups have converted their half of it.
// Each item writes its unnormalised O with (max, sum); the combine kernel
// merges the splits (all in log2 units).
#include <algorithm>
#include <cmath>

#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

struct AttnTc8Cfg {
  int stages;         // raw chunk stages
  uint32_t idesc_s;   // kind::f16 f16 x f16, M = 128, N = 128
  uint32_t idesc_o;   // kind::f16 f16 x f16, M = 128, N = d
  float scale_log2;   // log2(e) / sqrt(d)
};

constexpr int kA8Threads = 384;
constexpr int kA8SmThreads = 256;           // warps 2..9
constexpr int kA8CvThreads = 64;            // warps 10, 11
constexpr int kA8CvTid0 = 320;
constexpr int kA8SmBar = 3;                 // named barrier of the softmax warps
constexpr int kA8D = 128;                   // head dim (one 128-byte e4m3 row)
constexpr int kA8Atom = 128 * 128;          // 128 rows x 128 B (one K-atom of 64 f16)
constexpr int kA8KPage = kPage * kA8D;      // 8 KB of K codes per page
constexpr int kA8VPage = kA8D * kPage;      // 8 KB of V^T codes per page
constexpr int kA8Raw = 2 * kA8KPage + 2 * kA8VPage + 4 * kPage * 4;   // + K and V scales of two pages
constexpr int kA8V16Page = kA8D * 128;      // f16 V^T page: d rows x 64 keys x 2 B
constexpr int kA8V16 = 2 * kA8V16Page;      // one chunk (two pages)
constexpr int kA8MaxStages = 3;
constexpr int kA8Ksc = 2 * kPage * 4;      // K scales of one chunk (bytes)
constexpr int kA8Chunk = 2 * kPage;
constexpr float kA8RescaleLog2 = 8.f;

// Two codes widened to f16 times 2^-8 (e4m3x2_to_f16x2_scaled, integer
// operations) times their scales times 2^8, each product in f32 (exact: 4 +
// 24 significant bits; the powers of two cancel exactly) rounded once to f16.
__device__ __forceinline__ uint32_t scaled_f16x2(uint32_t widened, float s0x256, float s1x256) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&widened));
  const __half2 r = __floats2half2_rn(f.x * s0x256, f.y * s1x256);
  return *reinterpret_cast<const uint32_t*>(&r);
}

__global__ void __launch_bounds__(kA8Threads, 1)
    attn_tc8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, AttnArgs a, AttnTc8Cfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geo& g = a.g;
  uint8_t* sQ = smem;                                   // 2 atoms: f16 queries
  uint8_t* sK16 = sQ + 2 * kA8Atom;                     // 2 atoms: f16 keys of one chunk
  uint8_t* sV16 = sK16 + 2 * kA8Atom;                   // 2 x f16 V^T of one chunk
  uint8_t* sRaw = sV16 + 2 * kA8V16;                    // stages x raw chunk (1024-aligned: swizzled TMA)
  float* sKsc = reinterpret_cast<float*>(sRaw + t.stages * kA8Raw);   // 3 x K scales of one chunk
  uint8_t* ctl = sRaw + t.stages * kA8Raw + 3 * kA8Ksc;
  uint64_t* rawfull = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* rawempty = rawfull + kA8MaxStages;
  uint64_t* k16full = rawempty + kA8MaxStages;
  uint64_t* v16full = k16full + 1;                      // [2]
  uint64_t* sfull = v16full + 2;                        // [2]
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
  for (int idx = threadIdx.x; idx < 2 * (128 - R) * 32; idx += kA8Threads) {
    const int atom = idx / ((128 - R) * 32), rem = idx % ((128 - R) * 32);
    reinterpret_cast<uint32_t*>(sQ + atom * kA8Atom + R * 128)[rem] = 0u;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&rawfull[s], 1);
      mbar_init(&rawempty[s], kA8CvThreads + kA8SmThreads);
    }
    mbar_init(k16full, kA8CvThreads);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&v16full[b], kA8SmThreads);
      mbar_init(&sfull[b], 1);
      mbar_init(&pfull[b], kA8SmThreads);
      mbar_init(&pvdone[b], 1);
    }
    mbar_init(qfull, 1);
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

  // the descriptor, page table and cached-context pages are read before the
  // launch wait, as in attn_tc.cu
  const int item = a.rd->perm[blockIdx.x];              // longest items launch first
  int s, kvh, k0, k1, ks;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1, &ks);
  const int n_pages = (k1 - k0 + kPage - 1) / kPage;
  const int n_chunks = (n_pages + 1) / 2;
  const int slot = a.rd->seq_slot[s];
  const int len = a.rd->len[s];
  auto pages_in = [&](int c) { return min(2, n_pages - 2 * c); };
  auto raw_of = [&](int c) { return sRaw + (c % t.stages) * kA8Raw; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      const uint64_t pol = policy_evict_first();
      const float* ksc = fp8_pool_scales(g, a.kpool);
      const float* vsc = fp8_pool_scales(g, a.vpool);
      // page j of the split: K codes at stage + (j&1) x 8 KB, V^T codes after
      // both K pages, then the K scales [2][64] and V scales [2][64]
      auto load_page = [&](int j) -> bool {
        const int w = j & 1;
        const int page = a.block_table[(long)slot * g.pages_per_seq + k0 / kPage + j];
        if (page < 0 || page >= g.max_pages) {
          atomicExch(a.err, DERR_BAD_PAGE);
          return false;
        }
        const long base = ((long)a.layer * g.max_pages + page) * g.Hkv + kvh;
        uint8_t* st = raw_of(j >> 1);
        uint64_t* bar = &rawfull[(j >> 1) % t.stages];
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
      // the first raw stages are free: announce them and fetch their
      // context-only pages before the launch wait (the pages holding this
      // round's block rows are written by the predecessor)
      const int pre = min(n_chunks, t.stages);
      for (int c = 0; c < pre; ++c) {
        mbar_arrive_expect_tx(&rawfull[c], chunk_bytes(c));
        for (int w = 0; w < pages_in(c); ++w) {
          const int j = 2 * c + w;
          if (k0 + (j + 1) * kPage <= len) ok = ok && load_page(j);
          else deferred[nd++] = j;
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      mbar_arrive_expect_tx(qfull, (uint32_t)(2 * R * 128));
      for (int at = 0; at < 2; ++at) tma_load_3d(sQ + at * kA8Atom, &tmQ, qfull, at * 64, kvh * g.G, s * kBlock);
      for (int i = 0; i < nd && ok; ++i) ok = load_page(deferred[i]);
      unsigned long long wraw = 0;   // traced: cycles waiting for a free raw stage
      for (int c = pre; c < n_chunks && ok; ++c) {
        const int st = c % t.stages;
        const unsigned long long w0 = a.trace ? trace_clock() : 0;
        if (!mbar_wait(&rawempty[st], ((c / t.stages) & 1) ^ 1, &flags[0])) {
          ok = false;
          break;
        }
        if (a.trace) wraw += trace_clock() - w0;
        mbar_arrive_expect_tx(&rawfull[st], chunk_bytes(c));
        for (int w = 0; w < pages_in(c) && ok; ++w) ok = load_page(2 * c + w);
      }
      trace_put(a.trace, blockIdx.x, 12, wraw);   // 12: producer cycles waiting for a free raw stage
      if (!ok) flags[0] = 1;
    }
  } else if (warp >= kA8CvTid0 / 32) {
    // ------------------------------------------------------------------ converters
    // They read only shared memory filled by the producer's copies, so they
    // start on the context pages fetched before the launch wait.  A failed
    // wait skips the work but keeps every barrier arrival.
    const int ct = threadIdx.x - kA8CvTid0;   // 0..63
    bool ok = true;
    unsigned long long wr = 0, wk = 0;   // traced: cycles waiting for raw data and the K operand
    for (int c = 0; c < n_chunks; ++c) {
      const uint8_t* raw = raw_of(c);
      const float* ssc = reinterpret_cast<const float*>(raw + 2 * kA8KPage + 2 * kA8VPage);
      // (1) the raw chunk has landed and S(c-1) is done reading the K operand
      unsigned long long w0 = a.trace ? trace_clock() : 0;
      bool got = ok && mbar_wait(&rawfull[c % t.stages], (c / t.stages) & 1, &flags[0]);
      unsigned long long w1 = a.trace ? trace_clock() : 0;
      if (got && c >= 1) got = mbar_wait(&sfull[(c - 1) & 1], ((c - 1) >> 1) & 1, &flags[0]);
      if (a.trace) {
        wr += w1 - w0;
        wk += trace_clock() - w1;
      }
      got = __all_sync(0xffffffffu, got);
      if (!got) ok = false;
      __syncwarp();
      // (2) K codes -> f16 (exact) and the K scales of the chunk into scale
      // buffer c % 3 (the softmax of chunk c-3 is done with it: S(c-1) was
      // issued after P V^T of chunk c-3, hence after its softmax).  Item
      // (page w, key rr, 16-code piece j): K operand row r = 64 w + rr, atom
      // j / 4, f16 pieces 2 (j % 4), +1.
      if (ok) {
        // (the K operand holds the codes' values times 2^-8: the scales
        // carry 2^8, exactly)
        float* ksc = sKsc + (c % 3) * (2 * kPage);
        for (int i = ct; i < 2 * kPage; i += kA8CvThreads) ksc[i] = ssc[i] * kW8Unscale;
        // four items in flight per thread (their loads and conversions
        // overlap; one at a time the chain is latency-bound)
#pragma unroll 4
        for (int it = ct; it < pages_in(c) * kPage * 8; it += kA8CvThreads) {
          const int w = it >> 9, rr = (it >> 3) & (kPage - 1), j = it & 7;
          const uint4 src = *reinterpret_cast<const uint4*>(raw + w * kA8KPage + rr * 128 + ((j ^ (rr & 7)) << 4));
          const uint32_t sw[4] = {src.x, src.y, src.z, src.w};
          uint32_t hv[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint2 f4 = e4m3x4_to_f16x4_scaled(sw[i]);   // exact, times 2^-8
            hv[2 * i] = f4.x;
            hv[2 * i + 1] = f4.y;
          }
          const int r = w * kPage + rr, cc = 2 * (j & 3);
          uint8_t* drow = sK16 + (j >> 2) * kA8Atom + r * 128;
          *reinterpret_cast<uint4*>(drow + ((cc ^ (r & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(drow + (((cc + 1) ^ (r & 7)) << 4)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(k16full);
      mbar_arrive(&rawempty[c % t.stages]);
    }
    if (ct == 0) {
      trace_put(a.trace, blockIdx.x, 8, wr);    // 8: converter cycles waiting for raw chunks
      trace_put(a.trace, blockIdx.x, 9, wk);    // 9: ... for the K operand (S of the chunk before)
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(qfull, 0, &flags[0]);
      tc_fence_after();
      trace_mark(a.trace, blockIdx.x, 2, c0);                   // 2: query tile ready
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK16);
      auto issue_s = [&](int c) {
        tc_fence_after();
        const uint32_t d_s = tmem + 128u + (uint32_t)((c & 1) * kA8Chunk);
        for (int kk = 0; kk < 8; ++kk) {
          const int at = kk >> 2;
          const uint64_t adv = (uint64_t)((kk & 3) * 32) >> 4;
          mma_bf16(d_s, desc_sw128(q_addr + at * kA8Atom) + adv, desc_sw128(k_addr + at * kA8Atom) + adv, t.idesc_s,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(&sfull[c & 1]);
      };
      // O += P(c) V(c)^T: P of key half h in columns [64h, 64h + 32) of S
      // buffer c&1 (two keys per column), V^T page h of V buffer c&1
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
      // dependency order: S(ns) once the K operand of chunk ns is converted
      // and S buffer ns&1 is free (PV(ns-2) issued); PV(np) once the softmax
      // warps published P and the converters the V operand of chunk np
      int ns = 0, np = 0;
      uint64_t t_last = globaltimer();
      while (ok && np < n_chunks) {
        bool prog = false;
        if (np < ns && mbar_try_wait(&pfull[np & 1], (np >> 1) & 1) &&
            mbar_try_wait(&v16full[np & 1], (np >> 1) & 1)) {
          issue_pv(np++);
          prog = true;
        }
        if (ns < n_chunks && ns <= np + 1 && mbar_try_wait(k16full, ns & 1)) {
          issue_s(ns++);
          prog = true;
        }
        if (prog) t_last = globaltimer();
        else if (flags[0] || globaltimer() - t_last > kWaitNs) ok = false;
      }
      if (!ok) flags[0] = 1;
      trace_mark(a.trace, blockIdx.x, 3, c0);                   // 3: last MMA issued
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ softmax warps
    pdl_wait();
    const int q = warp & 3;
    const int hg = (warp - 2) >> 2;              // key half of every chunk (and half of O's columns)
    const int r = 32 * q + lane;                 // query row of this thread
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t xcol = tmem + lane_base + 384u;
    const int ocols = kA8D / 2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    auto sm_sync = [&]() { asm volatile("barrier.sync %0, %1;" ::"r"(kA8SmBar), "r"(kA8SmThreads) : "memory"); };
    unsigned long long ws = 0, wv = 0;   // traced: cycles waiting for scores / for a free V operand
    const int st_ = threadIdx.x - 64;    // 0..255
    for (int c = 0; c < n_chunks; ++c) {
      // V^T codes x V scales -> f16 into V buffer c&1, once the raw chunk has
      // landed and P V^T of chunk c-2 (the buffer's last reader) is done.
      // Items: 16-key pieces (page, d row, piece); a warp reads 512
      // contiguous bytes and writes 8 whole 128-byte rows.
      {
        const uint8_t* raw = raw_of(c);
        const float* ssc = reinterpret_cast<const float*>(raw + 2 * kA8KPage + 2 * kA8VPage);
        const unsigned long long w1 = a.trace ? trace_clock() : 0;
        bool vok = ok && mbar_wait(&rawfull[c % t.stages], (c / t.stages) & 1, &flags[0]);
        if (vok && c >= 2) vok = mbar_wait(&pvdone[c & 1], ((c - 2) >> 1) & 1, &flags[0]);
        vok = __all_sync(0xffffffffu, vok);
        if (a.trace) wv += trace_clock() - w1;
        if (!vok) ok = false;
        __syncwarp();
        if (ok) {
          uint8_t* vdst = sV16 + (c & 1) * kA8V16;
          for (int it = st_; it < pages_in(c) * kA8D * 4; it += kA8SmThreads) {
            const int w = it >> 9, row = (it >> 2) & (kA8D - 1), pc = it & 3;
            const uint4 src = *reinterpret_cast<const uint4*>(raw + 2 * kA8KPage + w * kA8VPage + row * kPage + pc * 16);
            const float4* svp = reinterpret_cast<const float4*>(ssc + (2 + w) * kPage + pc * 16);
            const uint32_t sw[4] = {src.x, src.y, src.z, src.w};
            uint32_t hv[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 sv4 = svp[i];   // scales of keys 4i .. 4i+3 of the piece
              const uint2 f4 = e4m3x4_to_f16x4_scaled(sw[i]);
              hv[2 * i] = scaled_f16x2(f4.x, sv4.x * kW8Unscale, sv4.y * kW8Unscale);
              hv[2 * i + 1] = scaled_f16x2(f4.y, sv4.z * kW8Unscale, sv4.w * kW8Unscale);
            }
            uint8_t* drow = vdst + w * kA8V16Page + row * 128;
            *reinterpret_cast<uint4*>(drow + (((2 * pc) ^ (row & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4*>(drow + (((2 * pc + 1) ^ (row & 7)) << 4)) =
                make_uint4(hv[4], hv[5], hv[6], hv[7]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&v16full[c & 1]);
        mbar_arrive(&rawempty[c % t.stages]);
      }
      const unsigned long long w0 = a.trace ? trace_clock() : 0;
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sfull[c & 1], (c >> 1) & 1, &flags[0]));
      if (a.trace) ws += trace_clock() - w0;
      if (!got) ok = false;
      __syncwarp();
      tc_fence_after();
      float sc[kPage];
      const uint32_t sbase = tmem + lane_base + 128u + (uint32_t)((c & 1) * kA8Chunk + hg * kPage);
      const int kbase = k0 + c * kA8Chunk + hg * kPage;
      const int kc = min(kPage, k1 - kbase);   // valid keys of this half (may be <= 0)
      const int klo = ks - kbase;              // keys below the window start (first page only)
      // scores times their keys' scales (masked keys -inf; whole pages skip
      // the mask); the log2-domain scale goes into the maximum and exp2
      const float* sk = sKsc + (c % 3) * (2 * kPage) + hg * kPage;
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
      const float mj = t.scale_log2 * fmaxf(mh, tmem_ld1(xcol + (uint32_t)(2 * (c & 1) + (hg ^ 1))));
      if (!ok || flags[0]) {
        ok = false;
        mbar_arrive(&pfull[c & 1]);
        continue;
      }
      const bool need = mj > m_run + kA8RescaleLog2;
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
      // P = 2^(scale t - m) (f16 pairs) over this half's own scores; masked
      // keys (t = -inf) give exact zeros
      const float nm = -m_run;
      float lsum = 0.f;
      float pw[kPage / 2];
#pragma unroll
      for (int i = 0; i < kPage / 2; ++i) {
        const float p0 = ex2_fast(fmaf(sc[2 * i], t.scale_log2, nm));
        const float p1 = ex2_fast(fmaf(sc[2 * i + 1], t.scale_log2, nm));
        lsum += p0 + p1;
        const __half2 hp = __floats2half2_rn(p0, p1);
        pw[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&hp));
      }
      tmem_st32(sbase, pw);
      l_run += lsum;
      tc_fence_before();
      mbar_arrive(&pfull[c & 1]);
    }
    if (threadIdx.x == 64) {
      trace_put(a.trace, blockIdx.x, 10, wv);   // 10: softmax warps' cycles waiting for raw data / a free V operand
      trace_put(a.trace, blockIdx.x, 11, ws);   // 11: softmax cycles waiting for scores
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
  trace_exit_warp(a.trace, blockIdx.x);
  if (flags[0] && threadIdx.x == 0) atomicExch(a.err, DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t attn_tc8_smem_bytes(int stages) {
  return (size_t)4 * kA8Atom + 2 * kA8V16 + 3 * kA8Ksc + (size_t)stages * kA8Raw + 256 + 1024;
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
