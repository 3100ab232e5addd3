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
//
// e4m3 weights (w8) stream as one byte each, in 8 KB units.  The producer
// then fills a ring of raw slots (up to 16, fetched ahead of the MMA stages,
// which are fewer); eight more warps widen each unit to f16 in the MMA
// stage's swizzled layout (exact: every e4m3 value times 2^-8 is an f16
// value, and integer operations produce it; the row scales carry 2^8); one
// more warp loads each stage's operand planes (f16 hi/lo beside e4m3
// weights, as kind::f16 takes one type for both operands); the issuers take
// a stage once both are in.  The per-row scales multiply the sums as they
// are drained.  The MMA reads the widened 16 KB from shared memory, as for
// bf16 weights, so an e4m3 unit costs the tensor cores what a bf16 one does:
// the gain is HBM bytes and footprint, not MMA time.
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
  int raw_slots;     // w8: raw e4m3 slots after the stages
  int conv;          // w8: units widened at once (stages and raw_slots are multiples), 2 or 4
  uint32_t idesc;
};

constexpr int kTcThreads = 224;   // warps: 0 producer, 1..2 MMA issuers, 3..6 drain
constexpr int kDrainTid0 = 96;    // first drain thread (warp 3)
constexpr int kConvTid0 = 224;    // w8: first converter thread (warps 7..14)
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kXLoadWarp = (kConvTid0 + kConvThreads) / 32;   // w8: warp 15 loads the operand planes
constexpr int kTcThreadsW8 = kConvTid0 + kConvThreads + 32;
constexpr int kMaxIss = 2;
constexpr int kWTileBytes = kTileN * kTileK * 2;   // 16 KB
constexpr int kRawBytes = kTileN * kTileK;         // 8 KB of e4m3 codes
constexpr int kMaxRaw = 16;
constexpr int kCtlBytes = 512;
constexpr int kCtlBytesW8 = 1024;
constexpr int kXBox = 16;                           // operand rows per short TMA box
constexpr int kXBoxTall = 128;                      // operand rows per tall TMA box

// One CTA per SM with a deep ring: every stage it can hold is filled with
// weights before the programmatic-launch wait, so HBM keeps streaming while
// the small kernel before it finishes.
template <bool kFused, int kIss, bool kW8>
__global__ void __launch_bounds__(kW8 ? kTcThreadsW8 : kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXT, GemmArgs a,
                   TcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem + t.stages * t.stage_bytes;                 // w8: raw e4m3 slots
  uint8_t* ctl = raw + t.raw_slots * kRawBytes;
  // control block: TMEM address, flags, then the barriers (ctl_bytes)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl);
  volatile int* flags = reinterpret_cast<volatile int*>(ctl + 16);   // abort, last
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl + 32);   // w8: the operand planes only
  uint64_t* empty = full + t.stages;
  uint64_t* accfull = empty + t.stages;          // [issuer][buffer]
  uint64_t* accempty = accfull + 2 * kMaxIss;     // [issuer][buffer]
  uint64_t* wready = accempty + 2 * kMaxIss;      // w8: stage's weights widened [stages]
  uint64_t* rawfull = wready + t.stages;          // w8: [raw_slots]
  uint64_t* rawempty = rawfull + t.raw_slots;     // w8: [raw_slots]
  float* red = reinterpret_cast<float*>(ctl + (kW8 ? kCtlBytesW8 : kCtlBytes));   // O_TILE only

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
    if (kW8) {
      // one arrival per converter warp of the unit's group
      for (int s = 0; s < t.stages; ++s) mbar_init(&wready[s], kConvWarps / t.conv);
      for (int r = 0; r < t.raw_slots; ++r) {
        mbar_init(&rawfull[r], 1);
        mbar_init(&rawempty[r], kConvWarps / t.conv);
      }
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
  // the operand planes of the unit at column kx into stage st (128-row boxes
  // while they fit in the pass, then 16-row boxes, so the boxes tile exactly
  // nt rows of each plane)
  const int y_hi = a.e.tok_base, y_lo = t.x_row_lo + a.e.tok_base;
  auto load_x = [&](uint8_t* st, uint64_t* bar, int kx) {
    int r = 0;
    for (; r + kXBoxTall <= t.nt; r += kXBoxTall) {
      tma_load_2d(st + kWTileBytes + r * 128, &tmXT, bar, kx, y_hi + r);
      tma_load_2d(st + kWTileBytes + x_plane_bytes + r * 128, &tmXT, bar, kx, y_lo + r);
    }
    for (; r < t.nt; r += kXBox) {
      tma_load_2d(st + kWTileBytes + r * 128, &tmX, bar, kx, y_hi + r);
      tma_load_2d(st + kWTileBytes + x_plane_bytes + r * 128, &tmX, bar, kx, y_lo + r);
    }
  };
  const int kmax = p.kb * kTileK;

  if (kW8 && warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- producer (e4m3)
      // raw codes only; every slot is filled before the launch wait
      const uint64_t pol = policy_evict_first();
      const uint8_t* wsrc = static_cast<const uint8_t*>(a.W) + (size_t)u0 * kRawBytes;
      const int pre = min(n_units, t.raw_slots);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&rawfull[i], kRawBytes);
        bulk_load_hint(raw + i * kRawBytes, wsrc + (size_t)i * kRawBytes, kRawBytes, &rawfull[i], pol);
      }
      pdl_wait();
      pdl_launch_dependents();
      trace_mark(a.trace, blockIdx.x, 2, c0);               // 2: producer past the launch wait
      int rs = 0;
      uint32_t ph = 0;
      unsigned long long waited = 0;
      for (int i = pre; i < n_units; ++i) {
        const unsigned long long w0 = a.trace ? trace_clock() : 0;
        if (!mbar_wait(&rawempty[rs], ph, &flags[0])) {
          flags[0] = 1;
          break;
        }
        if (a.trace) waited += trace_clock() - w0;
        mbar_arrive_expect_tx(&rawfull[rs], kRawBytes);
        bulk_load_hint(raw + rs * kRawBytes, wsrc + (size_t)i * kRawBytes, kRawBytes, &rawfull[rs], pol);
        if (++rs == t.raw_slots) {
          rs = 0;
          ph ^= 1;
        }
      }
      trace_put(a.trace, blockIdx.x, 9, waited);            // 9: producer cycles waiting for free slots
    }
  } else if (kW8 && warp == kXLoadWarp) {
    // ---------------------------------------------- operand loader (e4m3)
    // the unit's operand planes into its stage once the stage is free
    if (lane == 0) {
      pdl_wait();   // the operand planes come from the kernel before
      for (int i = 0; i < n_units; ++i) {
        const int st = i % t.stages;
        if (i >= t.stages && !mbar_wait(&empty[st], (uint32_t)(i / t.stages - 1) & 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[st], 2 * x_plane_bytes);
        load_x(smem + st * t.stage_bytes, &full[st], ((u0 + i) % p.kb) * kTileK);
      }
    }
  } else if (kW8 && warp >= kConvTid0 / 32) {
    // ------------------------------------------------------ converters (e4m3)
    // The eight converter warps form conv groups (two or four warps each);
    // group g takes the units i = g, g + conv, ..., so conv units widen at
    // once, and raw slot i % raw_slots and stage i % stages always belong to
    // the same group (both counts are multiples of conv), which keeps every
    // barrier's waiters on one phase.  Warp h of a group widens rows
    // 32 q + lane for its share of q = 0..3: a row's four 16-code pieces
    // (stored at piece position p ^ ((r >> 1) & 3), so that a quarter-warp's
    // reads hit eight bank groups) become its eight 16-byte f16 chunks at
    // chunk position c ^ (r & 7), the 128-byte swizzle the MMA reads.  Widening
    // is ALU-bound (about four integer operations per f16 pair), so two warps
    // per SM sub-partition keep up with the stream.
    const int cw = warp - kConvTid0 / 32;
    const int g = cw % t.conv, per = kConvWarps / t.conv, hq = cw / t.conv;
    const int q0 = hq * 4 / per, q1 = (hq + 1) * 4 / per;
    unsigned long long t_raw = 0, t_cv = 0, t_fence = 0;   // traced: cycles waiting for codes / widening / fencing
    for (int i = g; i < n_units; i += t.conv) {
      const int rs = i % t.raw_slots, st = i % t.stages;
      const unsigned long long w0 = a.trace ? trace_clock() : 0;
      if (!mbar_wait(&rawfull[rs], (uint32_t)(i / t.raw_slots) & 1, &flags[0])) {
        flags[0] = 1;
        break;
      }
      const unsigned long long w1 = a.trace ? trace_clock() : 0;
      // stage st is free once the MMAs of its previous unit completed
      if (i >= t.stages && !mbar_wait(&empty[st], (uint32_t)(i / t.stages - 1) & 1, &flags[0])) {
        flags[0] = 1;
        break;
      }
      const unsigned long long w2 = a.trace ? trace_clock() : 0;
      (void)w1;
      uint8_t* sp = smem + st * t.stage_bytes;
      const unsigned long long w3 = w2;
#pragma unroll 2
      for (int q = q0; q < q1; ++q) {
        const int r = lane + 32 * q;
        const int kswz = (r >> 1) & 3, cswz = r & 7;
        const uint8_t* src = raw + rs * kRawBytes + r * 64;
        uint8_t* dst = sp + r * 128;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const uint4 c = *reinterpret_cast<const uint4*>(src + ((pc ^ kswz) * 16));
          // codes (b0 b1 b2 b3) of a word become f16 pairs (b0, b1), (b2, b3)
          uint4 o0, o1;
          o0.x = e4m3x2_to_f16x2_scaled(__byte_perm(c.x, 0u, 0x4140));
          o0.y = e4m3x2_to_f16x2_scaled(__byte_perm(c.x, 0u, 0x4342));
          o0.z = e4m3x2_to_f16x2_scaled(__byte_perm(c.y, 0u, 0x4140));
          o0.w = e4m3x2_to_f16x2_scaled(__byte_perm(c.y, 0u, 0x4342));
          o1.x = e4m3x2_to_f16x2_scaled(__byte_perm(c.z, 0u, 0x4140));
          o1.y = e4m3x2_to_f16x2_scaled(__byte_perm(c.z, 0u, 0x4342));
          o1.z = e4m3x2_to_f16x2_scaled(__byte_perm(c.w, 0u, 0x4140));
          o1.w = e4m3x2_to_f16x2_scaled(__byte_perm(c.w, 0u, 0x4342));
          *reinterpret_cast<uint4*>(dst + (((2 * pc) ^ cswz) * 16)) = o0;
          *reinterpret_cast<uint4*>(dst + (((2 * pc + 1) ^ cswz) * 16)) = o1;
        }
      }
      __syncwarp();
      const unsigned long long w4 = a.trace ? trace_clock() : 0;
      fence_proxy_async_smem();   // this lane's generic-proxy writes, seen by the MMA
      __syncwarp();               // every lane's rows written and its codes read
      if (a.trace) {
        t_raw += w1 - w0;
        t_cv += w4 - w3;
        t_fence += trace_clock() - w4;
      }
      if (lane == 0) {
        mbar_arrive(&wready[st]);
        mbar_arrive(&rawempty[rs]);
      }
    }
    if (cw == 0 && lane == 0 && a.omode == O_RED) {   // (O_TILE epilogues use 8, 10)
      trace_put(a.trace, blockIdx.x, 8, t_raw);      // 8: converter 0 cycles waiting for codes
      trace_put(a.trace, blockIdx.x, 10, t_cv);      // 10: converter 0 cycles widening
      trace_put(a.trace, blockIdx.x, 13, t_fence);   // 13: converter 0 cycles in the proxy fence
    }
  } else if (warp == 0) {
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
      int kx = (u0 % p.kb) * kTileK;                        // operand column of the next unit
      auto next_x = [&](uint8_t* st, uint64_t* bar) {
        load_x(st, bar, kx);
        kx += kTileK;
        if (kx == kmax) kx = 0;
      };
      for (int i = 0; i < pre; ++i) next_x(smem + i * t.stage_bytes, &full[i]);
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
        next_x(sp, &full[st]);
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
          if (!mbar_wait(&full[st], ph, &flags[0]) || (kW8 && !mbar_wait(&wready[st], ph, &flags[0]))) {
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
  } else if (warp < kConvTid0 / 32) {
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
          const float wsc = a.e.wscale ? kW8Unscale * a.e.wscale[T * kTileN + row] : 1.f;
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
  trace_exit_warp(a.trace, blockIdx.x);
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

// Bytes of the control block: TMEM address and flags (32), full / empty per
// stage, two accumulator barriers per issuer buffer, and for e4m3 weights a
// widened-weights barrier per stage and two per raw slot.
static int ctl_bytes_needed(int stages, int raw_slots, bool w8) {
  return 32 + 8 * (2 * stages + 4 * kMaxIss + (w8 ? stages + 2 * raw_slots : 0));
}

// Shared memory of a launch: stages, (e4m3) raw slots, control block, the
// tile epilogue's scratch (O_TILE only) and the 1024-byte alignment slack.
static size_t tc_smem_bytes(const TcCfg& t, bool w8, bool tile) {
  return (size_t)t.stages * t.stage_bytes + (size_t)t.raw_slots * kRawBytes + (w8 ? kCtlBytesW8 : kCtlBytes) +
         (tile ? kRedFloats * 4 : 0) + 1024;
}

void launch_gemm_tc(const GemmArgs& a, const void* tmap_x, cudaStream_t s) {
  TcCfg t{};
  t.nt = (a.e.n_tok + 15) / 16 * 16;
  t.stage_bytes = kWTileBytes + 2 * t.nt * 128;
  constexpr int kSmemUse = 225 * 1024;
  const bool tile = a.omode == O_TILE;
  const int fixed = (a.w8 ? kCtlBytesW8 : kCtlBytes) + (tile ? kRedFloats * 4 : 0);
  // the lo plane follows the hi plane in the stage, so for nt <= 128 one MMA
  // with N = 2*nt multiplies both (half the tcgen05.mma issues; the drain adds
  // the two column halves)
  const bool fused = 2 * t.nt <= 256;
  t.aw = fused ? 2 * t.nt : t.nt;
  // two issuers when both have two accumulator buffers in the 512 TMEM columns
  const int iss = fused && 4 * t.aw <= 512 ? 2 : 1;
  if (!a.w8) {
    // as many stages as the SM's shared memory holds (weights prefetched
    // before the launch wait)
    t.stages = std::max(2, std::min(12, (kSmemUse - fixed) / t.stage_bytes));
  } else {
    // conv units widen at once, each group with spg stages (so that it can
    // widen its next unit while the MMAs read the last one) and the same
    // number of raw slots or more; the rest of shared memory holds raw e4m3
    // slots, which is what streams ahead of the MMAs.  Stages and slots are
    // multiples of conv (and the stages of the issuers).  Four units at once
    // with two stages each for short passes; fewer for operand-heavy passes
    // of 128 or more token columns.
    t.raw_slots = 0;
    const int pref[4][2] = {{4, 2}, {4, 1}, {2, 2}, {2, 1}};
    for (int c = 0; c < 4 && t.raw_slots == 0; ++c) {
      const int conv = pref[c][0], stages = conv * pref[c][1];
      if (stages % iss) continue;
      const int room = kSmemUse - fixed - stages * t.stage_bytes;
      int raw_slots = room > 0 ? std::min(kMaxRaw, room / kRawBytes) : 0;
      raw_slots -= raw_slots % conv;
      if (raw_slots >= std::max(4, stages)) {
        t.conv = conv;
        t.stages = stages;
        t.raw_slots = raw_slots;
      }
    }
    if (t.raw_slots == 0) return;   // never for nt <= 256; the caller's cudaGetLastError sees no launch
  }
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
  // the control block holds its words and barriers (ctl_bytes_needed <= the
  // reserved block for every nt <= 256; checked, as an overflow would run
  // into the epilogue's scratch)
  if (ctl_bytes_needed(t.stages, a.w8 ? t.raw_slots : 0, a.w8) > (a.w8 ? kCtlBytesW8 : kCtlBytes)) return;
  t.x_row_lo = a.e.g.Mt;
  // bf16 x bf16, or f16 x f16 beside e4m3 weights (format code 0)
  t.idesc = a.w8 ? idesc_fmt0(kTileN, t.aw) : idesc_bf16(kTileN, t.aw);
  const size_t smem = tc_smem_bytes(t, a.w8, tile);
  static size_t attr_bytes[6] = {0, 0, 0, 0, 0, 0};
  const int var = (!fused ? 0 : (iss == 1 ? 1 : 2)) + (a.w8 ? 3 : 0);
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, GemmArgs, TcCfg);
  static const Kern kerns[6] = {gemm_tc_kernel<false, 1, false>, gemm_tc_kernel<true, 1, false>,
                                gemm_tc_kernel<true, 2, false>,  gemm_tc_kernel<false, 1, true>,
                                gemm_tc_kernel<true, 1, true>,   gemm_tc_kernel<true, 2, true>};
  const Kern kern = kerns[var];
  if (smem > attr_bytes[var]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;   // the launch below is skipped; the caller's cudaGetLastError reports it
    attr_bytes[var] = smem;
  }
  // tmap_x: the operand's [16-row, 128-row] box maps
  const CUtensorMap* mx = static_cast<const CUtensorMap*>(tmap_x);
  launch_pdl(kern, dim3(a.p.grid), dim3(a.w8 ? kTcThreadsW8 : kTcThreads), smem, s, mx[0], mx[1], a, t);
}

}  // namespace dfl
