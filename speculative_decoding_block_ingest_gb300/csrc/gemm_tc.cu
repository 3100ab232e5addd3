// gemm_tc.cu -- weight-streaming projection on the 5th-generation tensor cores.
//
// Swap-AB: a 128-row weight tile is the MMA's A operand (M = 128 output
// features) and the token rows are its N side (16 per sequence), so the
// weight dimension fills the tensor core while the few drafted rows ride
// along.  Stream-K over units of 64 K-columns spreads a projection over the
// CTAs.  One CTA of nine warps per SM:
//   warp 0 (one lane)  producer: weight blocks [128 x 64] (one contiguous
//                      16 KB bulk copy each, stored pre-swizzled) and the
//                      operand's hi/lo bf16 planes [N x 64] (TMA) into a ring
//                      of stages (the first stages' weights before the
//                      programmatic-launch wait, so they stream during the
//                      previous kernel's tail);
//   warps 1, 2 (one lane each)  MMA issuers: ring slot i goes to issuer
//                      i % kIss, which runs its 4 K-steps x (hi, lo)
//                      tcgen05.mma into its own TMEM accumulator (two
//                      buffers).  At N = 32 one issuing thread moves a 16 KB
//                      unit in ~290 ns on this GB300 and two overlap to
//                      ~180 ns, which is also what more issuers reach: the
//                      tensor-core path tops out near 90 GB/s per SM at 16
//                      tokens, so a projection needs most SMs to stream HBM
//                      at full rate;
//   warps 3..6         drain: add the issuers' finished accumulators out of TMEM and
//                      red.add them into a token-major destination, or (for
//                      the ingest's projections) take the stream-K ticket and,
//                      as the last arriver, run the fused tile epilogue.
// The operand is split into two bf16 planes (x = hi + lo) so the product is
// f32-accurate in the activation; weights are exact bf16.
#include <algorithm>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

struct TcCfg {
  int nt;            // token columns per MMA (multiple of 16, <= 256)
  int stages;
  int stage_bytes;
  int tmem_cols;
  int aw;            // accumulator columns: 2*nt when hi and lo ride in one MMA, else nt
  int x_row_lo;      // row of the lo plane in the operand map (= Mt)
  uint32_t idesc;
};

constexpr int kTcThreads = 224;   // warps: 0 producer, 1..2 MMA issuers, 3..6 drain
constexpr int kDrainTid0 = 96;    // first drain thread (warp 3)
constexpr int kMaxIss = 2;
constexpr int kWTileBytes = kTileN * kTileK * 2;   // 16 KB
constexpr int kXBox = 16;                           // operand rows per short TMA box
constexpr int kXBoxTall = 128;                      // operand rows per tall TMA box

// One CTA per SM with a deep ring: every stage it can hold is filled with
// weights before the programmatic-launch wait, so HBM keeps streaming while
// the small kernel before it finishes.
template <bool kFused, int kIss>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXT, GemmArgs a,
                   TcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctl = smem + t.stages * t.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* empty = full + t.stages;
  uint64_t* accfull = empty + t.stages;          // [issuer][buffer]
  uint64_t* accempty = accfull + 2 * kMaxIss;     // [issuer][buffer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2 * kMaxIss);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort, last
  float* red = reinterpret_cast<float*>(ctl + 512);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long c0 = 0;
  if (threadIdx.x == 0) trace_entry(a.trace, blockIdx.x, &c0);
  if (a.trace) {
    __shared__ unsigned long long c0_shared;
    if (threadIdx.x == 0) c0_shared = c0;
    __syncthreads();
    c0 = c0_shared;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2 * kMaxIss; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiThreads);
    }
    flags[0] = flags[1] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmX);
    if (t.nt >= kXBoxTall) tma_prefetch_map(&tmXT);
  }
  if (warp == 1) tmem_alloc(tmem_slot, t.tmem_cols);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 1, c0);   // 1: set-up done

  const Part p = a.p;
  const int c = blockIdx.x;
  const int u0 = p.start(c), u1 = p.start(c + 1);
  const int n_units = u1 - u0;
  const uint32_t x_plane_bytes = (uint32_t)t.nt * 128;
  const int* err = a.e.err;

  // The two single-thread loops below are latency-bound on their own scalar
  // work, so they keep it minimal: stage index and phase are stepped, not
  // divided out, and the descriptors are the base descriptor plus offsets.
  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      const uint64_t pol = policy_evict_first();
      const uint8_t* wsrc = static_cast<const uint8_t*>(a.W) + (size_t)u0 * kWTileBytes;
      const uint32_t bytes = kWTileBytes + 2 * x_plane_bytes;
      const int pre = min(n_units, t.stages);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], bytes);
        bulk_load_hint(smem + i * t.stage_bytes, wsrc + (size_t)i * kWTileBytes, kWTileBytes, &full[i], pol);
      }
      pdl_wait();
      // dependents may launch only once this kernel is past its own wait, so
      // at most two kernels overlap and everything older has completed
      pdl_launch_dependents();
      trace_mark(a.trace, blockIdx.x, 2, c0);               // 2: producer past the launch wait
      const int kmax = p.kb * kTileK;
      const int y_hi = a.e.tok_base, y_lo = t.x_row_lo + a.e.tok_base;
      int kx = (u0 % p.kb) * kTileK;                        // operand column of the next unit
      auto load_x = [&](uint8_t* st, uint64_t* bar) {
        // 128-row boxes while they fit in the pass, then 16-row boxes, so
        // the boxes tile exactly nt rows of each plane
        int r = 0;
        for (; r + kXBoxTall <= t.nt; r += kXBoxTall) {
          tma_load_2d(st + kWTileBytes + r * 128, &tmXT, bar, kx, y_hi + r);
          tma_load_2d(st + kWTileBytes + x_plane_bytes + r * 128, &tmXT, bar, kx, y_lo + r);
        }
        for (; r < t.nt; r += kXBox) {
          tma_load_2d(st + kWTileBytes + r * 128, &tmX, bar, kx, y_hi + r);
          tma_load_2d(st + kWTileBytes + x_plane_bytes + r * 128, &tmX, bar, kx, y_lo + r);
        }
        kx += kTileK;
        if (kx == kmax) kx = 0;
      };
      for (int i = 0; i < pre; ++i) load_x(smem + i * t.stage_bytes, &full[i]);
      int st = 0;
      uint32_t ph = 0;   // parity of the empty phase the next refill waits for
      unsigned long long waited = 0;   // traced: cycles spent waiting for a free stage
      for (int i = pre; i < n_units; ++i) {
        const unsigned long long w0 = a.trace ? trace_clock() : 0;
        if (!mbar_wait(&empty[st], ph, &flags[0])) {
          flags[0] = 1;
          break;
        }
        if (a.trace) waited += trace_clock() - w0;
        uint8_t* sp = smem + st * t.stage_bytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_load_hint(sp, wsrc + (size_t)i * kWTileBytes, kWTileBytes, &full[st], pol);
        load_x(sp, &full[st]);
        if (++st == t.stages) {
          st = 0;
          ph ^= 1;
        }
      }
      trace_put(a.trace, blockIdx.x, 9, waited);            // 9: producer cycles waiting for free stages
    }
  } else if (warp >= 1 && warp <= kMaxIss) {
    // ---------------------------------------------------------------- MMA issuers
    // kIss issuers split every segment's units (ring slot i to issuer
    // i % kIss), each into its own pair of TMEM accumulators; the drain adds
    // them.
    const int j = warp - 1;
    if (lane == 0 && j < kIss) {
      // descriptor start fields are address >> 4 (14 bits, shared memory
      // < 256 KB), so stage and K-step offsets add without carries
      const uint64_t d0 = desc_sw128(smem_u32(smem));
      const uint32_t dstage = (uint32_t)t.stage_bytes >> 4;
      constexpr uint32_t xo = kWTileBytes >> 4;
      const uint32_t lo = (kWTileBytes + x_plane_bytes) >> 4;
      const uint32_t idesc = t.idesc;
      int seg = 0, st = j % t.stages;
      uint32_t ph = (uint32_t)(j / t.stages) & 1;
      bool ok = true;
      unsigned long long wfull = 0, wacc = 0;   // traced: cycles waiting for stages / accumulators
      for (int u = u0; u < u1 && ok; ++seg) {
        const int T = u / p.kb;
        const int seg_end = min(u1, (T + 1) * p.kb);
        const int b = seg & 1, use = seg >> 1;
        const unsigned long long w1 = a.trace ? trace_clock() : 0;
        if (!mbar_wait(&accempty[2 * j + b], (use & 1) ^ 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        if (a.trace) wacc += trace_clock() - w1;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)((2 * j + b) * t.aw);
        // this issuer's units of the segment: ring slots i = u - u0 with i % kIss == j
        int k = 0;
        for (int uu = u + ((j - (u - u0)) % kIss + kIss) % kIss; uu < seg_end; uu += kIss, ++k) {
          const unsigned long long w2 = a.trace ? trace_clock() : 0;
          if (!mbar_wait(&full[st], ph, &flags[0])) {
            flags[0] = 1;
            ok = false;
            break;
          }
          if (a.trace) wfull += trace_clock() - w2;
          tc_fence_after();
          const uint64_t dw = d0 + (uint64_t)(st * dstage);
          // 4 K-steps of 16 (32 bytes = 2 descriptor units each)
          mma_bf16(d_tmem, dw, dw + xo, idesc, k > 0 ? 1u : 0u);
          if (!kFused) mma_bf16(d_tmem, dw, dw + lo, idesc, 1u);
#pragma unroll
          for (uint32_t kk = 2; kk < 8; kk += 2) {
            mma_bf16(d_tmem, dw + kk, dw + xo + kk, idesc, 1u);
            if (!kFused) mma_bf16(d_tmem, dw + kk, dw + lo + kk, idesc, 1u);
          }
          mma_commit(&empty[st]);
          st += kIss;
          if (st >= t.stages) {
            st -= t.stages;
            ph ^= 1;
          }
        }
        // every segment is committed, also one without units of this issuer
        if (ok) mma_commit(&accfull[2 * j + b]);
        u = seg_end;
      }
      if (j == 0) trace_mark(a.trace, blockIdx.x, 3, c0);       // 3: last MMA issued
      if (j == 0 && a.omode == O_RED) {                          // (O_TILE epilogues use 11..13)
        trace_put(a.trace, blockIdx.x, 11, wfull);              // 11: issuer 0 cycles waiting for full stages
        trace_put(a.trace, blockIdx.x, 12, wacc);               // 12: issuer 0 cycles waiting for a free accumulator
      }
    }
  } else {
    // ------------------------------------------------------------------ drain
    pdl_wait();
    const int et = threadIdx.x - kDrainTid0;
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int row = 32 * q + lane;          // tile row (output feature) of this thread
    // the thread's row of accumulator buffer b of issuer j, token columns
    // j0..j0+15 (hi + lo halves when fused), added into v
    auto acc_add_ld16 = [&](int jb, int j0, float* v) {
      const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(jb * t.aw + j0);
      float w[16];
      tmem_ld16(base, w);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] += w[e];
      if (kFused) {
        tmem_ld16(base + (uint32_t)t.nt, w);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] += w[e];
      }
    };
    int seg = 0;
    for (int u = u0; u < u1; ++seg) {
      const int T = u / p.kb;
      const int seg_end = min(u1, (T + 1) * p.kb);
      const int b = seg & 1, use = seg >> 1;
      const bool last_seg = seg_end == u1;
      // units of each issuer in this segment (ring slots i = uu - u0, issuer i % kIss)
      int nu[kMaxIss];
#pragma unroll
      for (int jj = 0; jj < kMaxIss; ++jj) {
        // slots i in [u - u0, seg_end - u0) with i % kIss == jj
        const int first = u + ((jj - (u - u0)) % kIss + kIss) % kIss;
        nu[jj] = jj < kIss && first < seg_end ? (seg_end - 1 - first) / kIss + 1 : 0;
      }
      // a failed wait skips the TMEM read but keeps every barrier arrival, so
      // no thread is left waiting at a named barrier
      bool got = true;
      for (int jj = 0; jj < kIss; ++jj)
        got = __all_sync(0xffffffffu, mbar_wait(&accfull[2 * jj + b], use & 1, &flags[0])) && got;
      if (!got) flags[0] = 1;
      if (et == 0 && last_seg) trace_mark(a.trace, blockIdx.x, 6, c0);   // 6: last accumulator ready
      __syncwarp();
      tc_fence_after();
      if (a.omode == O_RED) {
        if (got) {
          float* dcol = a.dst + (long)a.e.tok_base * a.dst_ld + T * kTileN + row;
          const float wsc = a.e.wscale ? a.e.wscale[T * kTileN + row] : 1.f;
          for (int j0 = 0; j0 < a.e.n_tok; j0 += 16) {
            float v[16] = {};
            for (int jj = 0; jj < kIss; ++jj)
              if (nu[jj] > 0) acc_add_ld16(2 * jj + b, j0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j0 + j < a.e.n_tok)
                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dcol + (long)(j0 + j) * a.dst_ld), "f"(v[j] * wsc)
                             : "memory");
          }
        }
        tc_fence_before();
        for (int jj = 0; jj < kIss; ++jj) mbar_arrive(&accempty[2 * jj + b]);
      } else {
        float* acc_tile = a.acc + (long)T * kTileN * t.nt;
        if (got) {
          for (int j0 = 0; j0 < a.e.n_tok; j0 += 16) {
            float v[16] = {};
            for (int jj = 0; jj < kIss; ++jj)
              if (nu[jj] > 0) acc_add_ld16(2 * jj + b, j0, v);
            acc_add16(acc_tile + (long)row * t.nt, j0, a.e.n_tok, v);
          }
        }
        tc_fence_before();
        for (int jj = 0; jj < kIss; ++jj) mbar_arrive(&accempty[2 * jj + b]);
        __threadfence();
        epi_sync();
        if (et == 0) {
          const int c_lo = p.owner(T * p.kb), c_hi = p.owner((T + 1) * p.kb - 1);
          const int old = atomicAdd(a.counters + T, 1);
          flags[1] = (old == c_hi - c_lo);
        }
        epi_sync();
        if (flags[1]) {
          __threadfence();
          tile_epilogue(a.e, T, acc_tile, t.nt, red, et, last_seg ? a.trace : nullptr, blockIdx.x, c0);
          if (et == 0) a.counters[T] = 0;
          if (et == 0) trace_mark(a.trace, blockIdx.x, last_seg ? 10 : 8, c0);   // 10/8: tile epilogue done
        }
      }
      u = seg_end;
    }
    if (et == 0) trace_mark(a.trace, blockIdx.x, 4, c0);        // 4: drain loop done
  }
  __syncwarp();   // role lanes rejoin their warp before the CTA barrier
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 5, c0);  // 5: all roles done
  if (threadIdx.x == kDrainTid0) trace_mark(a.trace, blockIdx.x, 7, c0);
  if (threadIdx.x == 0) trace_exit(a.trace, blockIdx.x);
  if (flags[0] && threadIdx.x == 0) atomicExch(const_cast<int*>(err), DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, t.tmem_cols);
  }
}

// ------------------------------------------------------------------ host side
static int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

size_t gemm_tc_smem_bytes(int nt, int stages) {
  const int stage_bytes = kWTileBytes + 2 * nt * 128;
  return (size_t)stages * stage_bytes + 512 + kRedFloats * 4 + 1024;
}

void launch_gemm_tc(const GemmArgs& a, const void* tmap_x, cudaStream_t s) {
  TcCfg t{};
  t.nt = (a.e.n_tok + 15) / 16 * 16;
  t.stage_bytes = kWTileBytes + 2 * t.nt * 128;
  // as many stages as the SM's shared memory holds (weights prefetched before
  // the launch wait)
  t.stages = std::max(2, std::min(12, (225 * 1024 - 512 - kRedFloats * 4) / t.stage_bytes));
  // the lo plane follows the hi plane in the stage, so for nt <= 128 one MMA
  // with N = 2*nt multiplies both (half the tcgen05.mma issues; the drain adds
  // the two column halves)
  const bool fused = 2 * t.nt <= 256;
  t.aw = fused ? 2 * t.nt : t.nt;
  // two issuers when both have two accumulator buffers in the 512 TMEM columns
  const int iss = fused && 4 * t.aw <= 512 ? 2 : 1;
  // every stage belongs to one issuer (slot i goes to issuer i % iss and
  // stage i % stages), so the stage count is a multiple of the issuers:
  // otherwise a stage alternates between issuers, and one of them could wait
  // for the stage's next phase while the current one is still open, which
  // the phase parity cannot tell from the phase before it
  t.stages -= t.stages % iss;
  t.tmem_cols = pow2_at_least(2 * iss * t.aw);   // [issuer][buffer] accumulators
  // nt <= 256 per pass keeps this within an SM's 512 columns (fused: aw <= 256
  // and more issuers only while they fit; unfused: aw = nt <= 256); a larger
  // request would fault tcgen05.alloc, so it is never launched
  if (t.tmem_cols > 512 || t.stages < iss) return;
  t.x_row_lo = a.e.g.Mt;
  t.idesc = idesc_bf16(kTileN, t.aw);
  const size_t smem = gemm_tc_smem_bytes(t.nt, t.stages);
  static size_t attr_bytes[3] = {0, 0, 0};
  const int var = !fused ? 0 : (iss == 1 ? 1 : 2);
  auto kern = var == 0 ? gemm_tc_kernel<false, 1> : (var == 1 ? gemm_tc_kernel<true, 1> : gemm_tc_kernel<true, 2>);
  if (smem > attr_bytes[var]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;   // the launch below is skipped; the caller's cudaGetLastError reports it
    attr_bytes[var] = smem;
  }
  // tmap_x: the operand's [16-row, 128-row] box maps
  const CUtensorMap* mx = static_cast<const CUtensorMap*>(tmap_x);
  launch_pdl(kern, dim3(a.p.grid), dim3(kTcThreads), smem, s, mx[0], mx[1], a, t);
}

}  // namespace dfl
