// gemm_tt.cu -- token-tiled projection for rounds of many block rows.
//
// The weight-streaming projection (gemm_tc.cu) puts the weights on the MMA's
// M side and the few drafted rows on N; past 64 rows its operand planes
// outweigh the weights four to one per unit and the stages no longer fit
// shared memory deeply enough to stream.  Here the roles follow the data: a
// tile is 128 token rows (M, the operand's hi and lo bf16 planes as two A
// operands, loaded by TMA) by 256 output features (N, the two stacked 16 KB
// weight blocks of two 128-row tiles as B), accumulated over K in TMEM.
// Stream-K runs over units (token tile, feature tile, 64-column K step), K
// innermost, feature tile outermost, so that CTAs working on the same
// feature tile at once share its weights through L2 and every weight byte
// comes from HBM once per projection.  One CTA of six warps per SM:
//   warp 0 (one lane)  producer: per unit the two weight blocks (bulk copies,
//                      the first stages before the programmatic-launch wait)
//                      and the unit's 128 x 64 hi and lo operand boxes (TMA);
//   warp 1 (one lane)  MMA issuer: 4 K-steps x (hi, lo) tcgen05.mma of
//                      M = 128, N = 256 into one of two TMEM accumulators
//                      (256 columns each);
//   (e4m3 weights: warp 0 streams the codes, 8 KB per 128-row block, into a
//   ring of raw slots; warps 7..14 widen each unit's two blocks to f16 times
//   2^-8 into the stage (integer operations, exact; the row scales carry the
//   2^8); warp 6 loads the operand boxes; the operand planes are then f16.)
//   warps 2..5         drain: each warp reads its 32 token rows out of TMEM
//                      32 features at a time, turns the 32 x 32 block through
//                      shared memory and red.adds it as 16-byte vectors, four
//                      rows' 128 contiguous bytes per warp instruction
//                      instead of 32 rows' scattered words.
#include <algorithm>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kTtThreads = 192;          // warps: 0 producer, 1 issuer, 2..5 drain
constexpr int kTtXWarp = 6;              // e4m3: operand loader
constexpr int kTtConvWarp0 = 7;          // e4m3: converters 7..14
constexpr int kTtConvWarps = 8;
constexpr int kTtThreadsW8 = 32 * (kTtConvWarp0 + kTtConvWarps);   // 480
constexpr int kTtM = 128;                // token rows per tile
constexpr int kTtN = 2 * kTileN;         // output features per tile
constexpr int kTtABytes = kTtM * kTileK * 2;            // one operand plane box: 16 KB
constexpr int kTtBBytes = 2 * kTileN * kTileK * 2;      // two weight blocks: 32 KB
constexpr int kTtStageBytes = 2 * kTtABytes + kTtBBytes;   // 64 KB
constexpr int kTtStages = 3;
constexpr int kTtStagesW8 = 2;
constexpr int kTtRawBytes = 2 * kTileN * kTileK;   // e4m3 codes of a unit's two blocks: 16 KB
constexpr int kTtRawSlots = 4;
constexpr int kTtCtlBytes = 512;
constexpr int kTtTurnFloats = 32 * 33;   // a drain warp's 32 x 32 block, rows padded against bank conflicts

struct TtCfg {
  int n_tt, n_ft;      // token tiles, feature tiles
  uint32_t idesc;
};

template <bool kW8>
__global__ void __launch_bounds__(kW8 ? kTtThreadsW8 : kTtThreads, 1)
    gemm_tt_kernel(const __grid_constant__ CUtensorMap tmX, GemmArgs a, TtCfg t) {
  constexpr int S = kW8 ? kTtStagesW8 : kTtStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem + S * kTtStageBytes;                        // e4m3: [kTtRawSlots][kTtRawBytes]
  uint8_t* ctl = raw + (kW8 ? kTtRawSlots * kTtRawBytes : 0);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl);
  volatile int* flags = reinterpret_cast<volatile int*>(ctl + 16);   // abort
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl + 32);   // e4m3: the operand boxes only
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;            // [2]
  uint64_t* accempty = accfull + 2;         // [2]
  uint64_t* wready = accempty + 2;          // e4m3: [S] the stage's weights widened
  uint64_t* rawfull = wready + S;           // e4m3: [kTtRawSlots]
  uint64_t* rawempty = rawfull + kTtRawSlots;
  float* turn = reinterpret_cast<float*>(ctl + kTtCtlBytes);   // [4 drain warps][kTtTurnFloats]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long c0 = 0;
  if (threadIdx.x == 0) trace_entry(a.trace, blockIdx.x, &c0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if (kW8) mbar_init(&wready[s], kTtConvWarps);
    }
    if (kW8)
      for (int r = 0; r < kTtRawSlots; ++r) {
        mbar_init(&rawfull[r], 1);
        mbar_init(&rawempty[r], kTtConvWarps);
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiThreads);
    }
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const Part p = a.p;          // p.kb K steps per tile; tiles ordered (feature tile, token tile)
  const int u0 = p.start(blockIdx.x), u1 = p.start(blockIdx.x + 1);
  const int n_units = u1 - u0;

  auto load_x = [&](int u, uint8_t* st, uint64_t* bar) {
    const int tile = u / p.kb, k = u % p.kb, tt = tile % t.n_tt;
    const int y = a.e.tok_base + tt * kTtM;
    tma_load_2d(st, &tmX, bar, k * kTileK, y);                          // hi plane rows
    tma_load_2d(st + kTtABytes, &tmX, bar, k * kTileK, a.e.g.Mt + y);   // lo plane rows
  };
  if (kW8 && warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer (e4m3)
      // the codes of unit u: blocks (2 ft, k) and (2 ft + 1, k), 8 KB each
      const uint8_t* W = static_cast<const uint8_t*>(a.W);
      auto load_codes = [&](int u, int rs) {
        const int tile = u / p.kb, k = u % p.kb, ft = tile / t.n_tt;
        const size_t blk = (size_t)(2 * ft) * p.kb + k;
        mbar_arrive_expect_tx(&rawfull[rs], kTtRawBytes);
        bulk_load(raw + rs * kTtRawBytes, W + blk * (kTtRawBytes / 2), kTtRawBytes / 2, &rawfull[rs]);
        bulk_load(raw + rs * kTtRawBytes + kTtRawBytes / 2, W + (blk + p.kb) * (kTtRawBytes / 2), kTtRawBytes / 2,
                  &rawfull[rs]);
      };
      const int pre = min(n_units, kTtRawSlots);
      for (int i = 0; i < pre; ++i) load_codes(u0 + i, i);
      pdl_wait();
      pdl_launch_dependents();
      for (int i = pre; i < n_units; ++i) {
        const int rs = i % kTtRawSlots;
        if (!mbar_wait(&rawempty[rs], (uint32_t)(i / kTtRawSlots - 1) & 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        load_codes(u0 + i, rs);
      }
    }
  } else if (kW8 && warp == kTtXWarp) {
    if (lane == 0) {
      // ---------------------------------------------- operand loader (e4m3)
      pdl_wait();   // the operand planes come from the kernel before
      for (int i = 0; i < n_units; ++i) {
        const int st = i % S;
        if (i >= S && !mbar_wait(&empty[st], (uint32_t)(i / S - 1) & 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[st], 2 * kTtABytes);
        load_x(u0 + i, smem + st * kTtStageBytes, &full[st]);
      }
    }
  } else if (kW8 && warp >= kTtConvWarp0) {
    // ------------------------------------------------------ converters (e4m3)
    // warp w widens rows 32 (w % 4) + lane of block w / 4 of each unit: the
    // row's four 16-code pieces (piece p at piece position p ^ ((r >> 1) & 3))
    // become its eight 16-byte f16 chunks at chunk position c ^ (r & 7), the
    // 128-byte swizzle of the B operand (block 1's rows follow block 0's)
    const int cw = warp - kTtConvWarp0, blk = cw >> 2, r = 32 * (cw & 3) + lane;
    const int kswz = (r >> 1) & 3, cswz = r & 7;
    for (int i = 0; i < n_units; ++i) {
      const int rs = i % kTtRawSlots, st = i % S;
      if (!mbar_wait(&rawfull[rs], (uint32_t)(i / kTtRawSlots) & 1, &flags[0]) ||
          (i >= S && !mbar_wait(&empty[st], (uint32_t)(i / S - 1) & 1, &flags[0]))) {
        flags[0] = 1;
        break;
      }
      const uint8_t* src = raw + rs * kTtRawBytes + blk * (kTtRawBytes / 2) + r * 64;
      uint8_t* dst = smem + st * kTtStageBytes + 2 * kTtABytes + blk * (kTtBBytes / 2) + r * 128;
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const uint4 c = *reinterpret_cast<const uint4*>(src + ((pc ^ kswz) * 16));
        const uint2 w0 = e4m3x4_to_f16x4_scaled(c.x), w1 = e4m3x4_to_f16x4_scaled(c.y);
        const uint2 w2 = e4m3x4_to_f16x4_scaled(c.z), w3 = e4m3x4_to_f16x4_scaled(c.w);
        *reinterpret_cast<uint4*>(dst + (((2 * pc) ^ cswz) * 16)) = make_uint4(w0.x, w0.y, w1.x, w1.y);
        *reinterpret_cast<uint4*>(dst + (((2 * pc + 1) ^ cswz) * 16)) = make_uint4(w2.x, w2.y, w3.x, w3.y);
      }
      fence_proxy_async_smem();   // this lane's generic-proxy writes, seen by the MMA
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&wready[st]);
        mbar_arrive(&rawempty[rs]);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      const uint8_t* W = static_cast<const uint8_t*>(a.W);
      auto load_w = [&](int u, uint8_t* st, uint64_t* bar) {
        const int tile = u / p.kb, k = u % p.kb, ft = tile / t.n_tt;
        const size_t blk = (size_t)(2 * ft) * p.kb + k;   // block (2 ft, k), then (2 ft + 1, k)
        bulk_load(st + 2 * kTtABytes, W + blk * (kTtBBytes / 2), kTtBBytes / 2, bar);
        bulk_load(st + 2 * kTtABytes + kTtBBytes / 2, W + (blk + p.kb) * (kTtBBytes / 2), kTtBBytes / 2, bar);
      };
      const int pre = min(n_units, S);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], kTtStageBytes);
        load_w(u0 + i, smem + i * kTtStageBytes, &full[i]);
      }
      pdl_wait();
      pdl_launch_dependents();
      trace_mark(a.trace, blockIdx.x, 2, c0);               // 2: producer past the launch wait
      for (int i = 0; i < pre; ++i) load_x(u0 + i, smem + i * kTtStageBytes, &full[i]);
      int st = 0;
      uint32_t ph = 0;
      for (int i = pre; i < n_units; ++i) {
        if (!mbar_wait(&empty[st], ph, &flags[0])) {
          flags[0] = 1;
          break;
        }
        uint8_t* sp = smem + st * kTtStageBytes;
        mbar_arrive_expect_tx(&full[st], kTtStageBytes);
        load_w(u0 + i, sp, &full[st]);
        load_x(u0 + i, sp, &full[st]);
        if (++st == S) {
          st = 0;
          ph ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint64_t d0 = desc_sw128(smem_u32(smem));
      constexpr uint32_t dstage = (uint32_t)kTtStageBytes >> 4;
      constexpr uint32_t lo = (uint32_t)kTtABytes >> 4;
      constexpr uint32_t wo = (uint32_t)(2 * kTtABytes) >> 4;
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      int seg = 0;
      for (int u = u0; u < u1 && ok; ++seg) {
        const int seg_end = min(u1, (u / p.kb + 1) * p.kb);
        const int b = seg & 1, use = seg >> 1;
        if (!mbar_wait(&accempty[b], (use & 1) ^ 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(b * kTtN);
        for (int k = 0; u < seg_end; ++u, ++k) {
          if (!mbar_wait(&full[st], ph, &flags[0]) || (kW8 && !mbar_wait(&wready[st], ph, &flags[0]))) {
            flags[0] = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ds = d0 + (uint64_t)(st * dstage);
#pragma unroll
          for (uint32_t kk = 0; kk < 8; kk += 2) {
            mma_bf16(d_tmem, ds + kk, ds + wo + kk, t.idesc, (k > 0 || kk > 0) ? 1u : 0u);
            mma_bf16(d_tmem, ds + lo + kk, ds + wo + kk, t.idesc, 1u);
          }
          mma_commit(&empty[st]);
          if (++st == S) {
            st = 0;
            ph ^= 1;
          }
        }
        if (ok) mma_commit(&accfull[b]);
      }
      trace_mark(a.trace, blockIdx.x, 3, c0);                   // 3: last MMA issued
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------------ drain
    pdl_wait();
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    int seg = 0;
    for (int u = u0; u < u1; ++seg) {
      const int tile = u / p.kb;
      const int seg_end = min(u1, (tile + 1) * p.kb);
      const int b = seg & 1, use = seg >> 1;
      const int ft = tile / t.n_tt, tt = tile % t.n_tt;
      const bool got = __all_sync(0xffffffffu, mbar_wait(&accfull[b], use & 1, &flags[0]));
      if (!got) flags[0] = 1;
      __syncwarp();
      tc_fence_after();
      if (got) {
        const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * kTtN);
        float* tb = turn + (warp - 2) * kTtTurnFloats;
        const int tok0 = tt * kTtM + 32 * q;                 // the warp's first token row (within the pass)
        const int rows = min(32, a.e.n_tok - tok0);          // its rows that exist
        // lane l adds features 4 (l % 8) .. + 3 of row r + l / 8 as one
        // 16-byte red.add: a warp instruction covers four rows' 128 bytes
        const int rl = lane >> 3, c4 = 4 * (lane & 7);
        float* dst0 = a.dst + (long)(a.e.tok_base + tok0 + rl) * a.dst_ld + ft * kTtN + c4;
        // the CTAs sharing a tile drain together: each starts at another
        // 32-feature chunk, so their simultaneous red.adds hit other lines
        for (int jj = 0; jj < kTtN / 32; ++jj) {
          const int j0 = ((jj + blockIdx.x) & (kTtN / 32 - 1)) * 32;
          float v[32];
          tmem_ld32(base + (uint32_t)j0, v);                 // warp-wide: lane = row, v = 32 features
#pragma unroll
          for (int j = 0; j < 32; ++j) tb[lane * 33 + j] = v[j];
          __syncwarp();
          // e4m3: the lane's four features' row scales (times 2^8)
          float4 sc = make_float4(1.f, 1.f, 1.f, 1.f);
          if (kW8) {
            sc = __ldg(reinterpret_cast<const float4*>(a.e.wscale + ft * kTtN + j0 + c4));
            sc = make_float4(sc.x * kW8Unscale, sc.y * kW8Unscale, sc.z * kW8Unscale, sc.w * kW8Unscale);
          }
          for (int r = 0; r + rl < rows; r += 4) {
            const float* src = tb + (r + rl) * 33 + c4;
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst0 + (long)r * a.dst_ld + j0),
                         "f"(src[0] * sc.x), "f"(src[1] * sc.y), "f"(src[2] * sc.z), "f"(src[3] * sc.w)
                         : "memory");
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(&accempty[b]);
      u = seg_end;
    }
  }
  __syncwarp();
  __syncthreads();
  trace_exit_warp(a.trace, blockIdx.x);
  if (flags[0] && threadIdx.x == 0) atomicExch(a.e.err, DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool gemm_tt_fits(const GemmArgs& a) {
  return a.omode == O_RED && a.N % kTtN == 0 && a.K % kTileK == 0 && a.e.n_tok > 64;
}

int gemm_tt_units(const GemmArgs& a) {
  const int n_tt = (a.e.n_tok + kTtM - 1) / kTtM;
  return n_tt * (a.N / kTtN) * (a.K / kTileK);
}

void launch_gemm_tt(const GemmArgs& a, const void* tmap_x_tall, cudaStream_t s) {
  TtCfg t{};
  t.n_tt = (a.e.n_tok + kTtM - 1) / kTtM;
  t.n_ft = a.N / kTtN;
  // bf16 x bf16, or f16 x f16 beside e4m3 weights (format code 0)
  t.idesc = a.w8 ? idesc_fmt0(kTtM, kTtN) : idesc_bf16(kTtM, kTtN);
  const size_t smem = a.w8 ? (size_t)kTtStagesW8 * kTtStageBytes + (size_t)kTtRawSlots * kTtRawBytes + kTtCtlBytes +
                                 4 * kTtTurnFloats * 4 + 1024
                           : (size_t)kTtStages * kTtStageBytes + kTtCtlBytes + 4 * kTtTurnFloats * 4 + 1024;
  static bool attr[2] = {false, false};
  auto kern = a.w8 ? gemm_tt_kernel<true> : gemm_tt_kernel<false>;
  if (!attr[a.w8]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;   // the launch below is skipped; the caller's cudaGetLastError reports it
    attr[a.w8] = true;
  }
  launch_pdl(kern, dim3(a.p.grid), dim3(a.w8 ? kTtThreadsW8 : kTtThreads), smem, s,
             *static_cast<const CUtensorMap*>(tmap_x_tall), a, t);
}

}  // namespace dfl
