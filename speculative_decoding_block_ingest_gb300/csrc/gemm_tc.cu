// gemm_tc.cu -- weight-streaming projection on the 5th-generation tensor cores.
//
// Swap-AB: a 128-row weight tile is the MMA's A operand (M = 128 output
// features) and the token rows are its N side (16 per sequence), so the
// weight dimension fills the tensor core while the few drafted rows ride
// along.  One CTA per SM, three roles:
//   warp 0 (one lane)  TMA producer: weight tile [128 x 64] and the operand's
//                      hi and lo bf16 planes [N x 64] into a ring of stages;
//                      the first stages' weight loads are issued before the
//                      programmatic-launch wait, so they overlap the tail of
//                      the previous kernel;
//   warp 1 (one lane)  MMA issuer: per 64-column unit, 4 K-steps x (hi, lo)
//                      tcgen05.mma into a TMEM accumulator (two buffers);
//   warps 2..5         epilogue: TMEM -> f32 partial, stream-K arrival, and
//                      for the last arriver the tile's fused epilogue.
// The operand is split in two bf16 planes (x = hi + lo) so the product is
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
  int x_row_lo;      // row of the lo plane in the operand map (= Mt)
  uint32_t idesc;
};

constexpr int kTcThreads = 192;
constexpr int kWTileBytes = kTileN * kTileK * 2;   // 16 KB
constexpr int kXBox = 16;                           // operand rows per TMA box

__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, GemmArgs a,
                   TcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctl = smem + t.stages * t.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* empty = full + t.stages;
  uint64_t* accfull = empty + t.stages;
  uint64_t* accempty = accfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort, last, c_lo, c_hi
  float* red = reinterpret_cast<float*>(ctl + 512);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiThreads);
    }
    flags[0] = flags[1] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, t.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  const Part p = a.p;
  const int c = blockIdx.x;
  const int u0 = p.start(c), u1 = p.start(c + 1);
  const int n_units = u1 - u0;
  const uint32_t x_plane_bytes = (uint32_t)t.nt * 128;
  const int* err = a.e.err;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = kWTileBytes + 2 * x_plane_bytes;
      auto load_x = [&](int i, int u) {
        uint8_t* st = smem + (i % t.stages) * t.stage_bytes;
        const int kx = (u % p.kb) * kTileK;
        for (int r = 0; r < t.nt; r += kXBox) {
          tma_load_2d(st + kWTileBytes + r * 128, &tmX, &full[i % t.stages], kx, a.e.tok_base + r);
          tma_load_2d(st + kWTileBytes + x_plane_bytes + r * 128, &tmX, &full[i % t.stages], kx,
                      t.x_row_lo + a.e.tok_base + r);
        }
      };
      const int pre = min(n_units, t.stages);
      for (int i = 0; i < pre; ++i) {
        const int u = u0 + i;
        mbar_arrive_expect_tx(&full[i], bytes);
        tma_load_2d_hint(smem + i * t.stage_bytes, &tmW, &full[i], (u % p.kb) * kTileK, (u / p.kb) * kTileN, pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) load_x(i, u0 + i);
      for (int i = pre; i < n_units; ++i) {
        const int s = i % t.stages;
        if (!mbar_wait(&empty[s], ((i / t.stages) & 1) ^ 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        const int u = u0 + i;
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d_hint(smem + s * t.stage_bytes, &tmW, &full[s], (u % p.kb) * kTileK, (u / p.kb) * kTileN, pol);
        load_x(i, u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      int i = 0, seg = 0;
      bool ok = true;
      for (int u = u0; u < u1 && ok; ++seg) {
        const int T = u / p.kb;
        const int seg_end = min(u1, (T + 1) * p.kb);
        const int b = seg & 1, use = seg >> 1;
        if (!mbar_wait(&accempty[b], (use & 1) ^ 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(b * t.nt);
        for (const int seg_start = u; u < seg_end; ++u, ++i) {
          const int s = i % t.stages;
          if (!mbar_wait(&full[s], (i / t.stages) & 1, &flags[0])) {
            flags[0] = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * t.stage_bytes);
          const uint64_t dw = desc_sw128(sa);
          const uint64_t dh = desc_sw128(sa + kWTileBytes);
          const uint64_t dl = desc_sw128(sa + kWTileBytes + x_plane_bytes);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            const uint64_t adv = (uint64_t)(kk * 32) >> 4;   // 16 bf16 = 32 bytes per K-step
            mma_bf16(d_tmem, dw + adv, dh + adv, t.idesc, (u > seg_start || kk > 0) ? 1u : 0u);
            mma_bf16(d_tmem, dw + adv, dl + adv, t.idesc, 1u);
          }
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&accfull[b]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue warps
    pdl_wait();
    const int et = threadIdx.x - 64;
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int row = 32 * q + lane;          // tile row (output feature) of this thread
    const long slot_elems = (long)a.e.g.Mt * kTileN;
    int seg = 0;
    for (int u = u0; u < u1; ++seg) {
      const int T = u / p.kb;
      const int seg_end = min(u1, (T + 1) * p.kb);
      const int b = seg & 1, use = seg >> 1;
      if (!mbar_wait(&accfull[b], use & 1, &flags[0])) {
        flags[0] = 1;
        break;
      }
      __syncwarp();
      tc_fence_after();
      float* dst = a.part + (long)(c + T) * slot_elems;
      for (int j0 = 0; j0 < a.e.n_tok; j0 += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * t.nt + j0), v);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j0 + j < a.e.n_tok) dst[(long)(j0 + j) * kTileN + row] = v[j];
      }
      tc_fence_before();
      mbar_arrive(&accempty[b]);
      __threadfence();
      epi_sync();
      if (et == 0) {
        const int c_lo = p.owner(T * p.kb), c_hi = p.owner((T + 1) * p.kb - 1);
        const int old = atomicAdd(a.counters + T, 1);
        flags[1] = (old == c_hi - c_lo);
        flags[2] = c_lo;
        flags[3] = c_hi;
      }
      epi_sync();
      if (flags[1]) {
        __threadfence();
        const int c_lo = flags[2], c_hi = flags[3];
        tile_epilogue(a.e, T, c_lo, c_hi, a.part, red, et);
        if (et == 0) a.counters[T] = 0;
      }
      u = seg_end;
    }
  }
  __syncthreads();
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
  return (size_t)stages * stage_bytes + 512 + kEpiTokChunk * (kTileN + 1) * 4 + 1024;
}

void launch_gemm_tc(const GemmArgs& a, const void* tmap_w, const void* tmap_x, cudaStream_t s) {
  TcCfg t{};
  t.nt = (a.e.n_tok + 15) / 16 * 16;
  t.stage_bytes = kWTileBytes + 2 * t.nt * 128;
  // ~100 KB per CTA lets the next kernel's CTA share the SM during the tail
  t.stages = std::max(2, std::min(8, (100 * 1024 - 512 - kEpiTokChunk * (kTileN + 1) * 4) / t.stage_bytes));
  t.tmem_cols = pow2_at_least(2 * t.nt);
  t.x_row_lo = a.e.g.Mt;
  t.idesc = idesc_bf16(kTileN, t.nt);
  const size_t smem = gemm_tc_smem_bytes(t.nt, t.stages);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    attr_set = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.p.grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const CUtensorMap* mw = static_cast<const CUtensorMap*>(tmap_w);
  const CUtensorMap* mx = static_cast<const CUtensorMap*>(tmap_x);
  cudaLaunchKernelEx(&cfg, gemm_tc_kernel, *mw, *mx, a, t);
}

}  // namespace dfl
