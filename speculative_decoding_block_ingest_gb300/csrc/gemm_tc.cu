// gemm_tc.cu -- weight-streaming projection on the 5th-generation tensor cores.
//
// Swap-AB: a 128-row weight tile is the MMA's A operand (M = 128 output
// features) and the token rows are its N side (16 per sequence), so the
// weight dimension fills the tensor core while the few drafted rows ride
// along.  Stream-K over units of 64 K-columns spreads every projection over
// all SMs.  One CTA of six warps per SM (two fit):
//   warp 0 (one lane)  TMA producer: weight tiles [128 x 64] into a ring of
//                      stages (the first stages before the programmatic-launch
//                      wait, so they stream during the previous kernel's tail),
//                      and for prepared operands their hi/lo bf16 planes;
//   warp 1 (one lane)  MMA issuer: per unit, 4 K-steps x (hi, lo) tcgen05.mma
//                      into a TMEM accumulator (two buffers);
//   warps 2..5         operand converters and drain: they build the operand's
//                      hi/lo planes in shared memory from f32 sources (the
//                      residual stream times a norm gain, or the SwiGLU of the
//                      gate/up accumulator), then move finished accumulators out
//                      of TMEM: red.add into a token-major destination, or the
//                      stream-K ticket and, for the last arriver, the fused
//                      tile epilogue.
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
  int x_row_lo;      // row of the lo plane in the operand map (= Mt)
  uint32_t idesc;
};

constexpr int kTcThreads = 192;
constexpr int kWTileBytes = kTileN * kTileK * 2;   // 16 KB
constexpr int kXBox = 16;                           // operand rows per TMA box

// Pack 8 floats into 8 bf16 hi parts and 8 bf16 lo parts (x = hi + lo).
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[2 * q], x[2 * q + 1]);
    const float2 af = __bfloat1622float2(a);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * q] - af.x, x[2 * q + 1] - af.y);
    h[q] = *reinterpret_cast<const uint32_t*>(&a);
    l[q] = *reinterpret_cast<const uint32_t*>(&b);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Build the hi/lo operand planes of one unit (K columns kx..kx+63) in the
// 128-byte-swizzled K-major layout, 16 token rows per pass: thread et owns
// row (et / 8) and 16-byte chunk (et % 8) of each pass.
__device__ __forceinline__ void convert_unit(const GemmArgs& a, const TcCfg& t, uint8_t* xh, uint8_t* xl, int kx,
                                             int et) {
  const int ch = et & 7;
  const int c8 = kx + ch * 8;
  float gn[8];
  if (a.xmode == X_FROM_H) {
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.xgain + c8));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.xgain + c8) + 1);
    gn[0] = g0.x; gn[1] = g0.y; gn[2] = g0.z; gn[3] = g0.w;
    gn[4] = g1.x; gn[5] = g1.y; gn[6] = g1.z; gn[7] = g1.w;
  }
  for (int r0 = 0; r0 < t.nt; r0 += 16) {
    const int r = r0 + (et >> 3);
    const int tok = a.e.tok_base + r;
    float x[8];
    if (r < a.e.n_tok) {
      if (a.xmode == X_FROM_H) {
        const float4* src = reinterpret_cast<const float4*>(a.xsrc + (long)tok * a.xsrc_ld + c8);
        const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
        x[0] = v0.x * gn[0]; x[1] = v0.y * gn[1]; x[2] = v0.z * gn[2]; x[3] = v0.w * gn[3];
        x[4] = v1.x * gn[4]; x[5] = v1.y * gn[5]; x[6] = v1.z * gn[6]; x[7] = v1.w * gn[7];
      } else {   // X_SWIGLU: gate/up tile kx/64 holds gate at +0..63, up at +64..127
        const long base = (long)tok * a.xsrc_ld + (kx / 64) * 128 + ch * 8;
        const float4* gp = reinterpret_cast<const float4*>(a.xsrc + base);
        const float4* up = reinterpret_cast<const float4*>(a.xsrc + base + 64);
        const float4 g0 = __ldcg(gp), g1 = __ldcg(gp + 1), u0 = __ldcg(up), u1 = __ldcg(up + 1);
        const float rs = a.xrs[tok];
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float gs = gv[q] * rs;
          x[q] = gs / (1.f + __expf(-gs)) * (uv[q] * rs);
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = 0.f;
    }
    uint4 hi, lo;
    split8(x, hi, lo);
    const int off = (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(xh + off) = hi;
    *reinterpret_cast<uint4*>(xl + off) = lo;
  }
}

// Staged conversion for passes of at most 16 tokens: the f32 sources of the
// next units are fetched into a small shared ring with cp.async while the
// current unit is converted, so the MMA never waits a full L2 round trip.
//   X_FROM_H slot: x [16][64] f32, gain [64]         (3 slots)
//   X_SWIGLU slot: gate [16][64], up [16][64], r [16] (2 slots)
constexpr int kStgFromHBytes = 16 * 64 * 4 + 64 * 4;
constexpr int kStgSwiBytes = 2 * 16 * 64 * 4 + 16 * 4;

__device__ __forceinline__ int stage_slots(int xmode) { return xmode == X_FROM_H ? 3 : 2; }

__device__ __forceinline__ void stage_issue(const GemmArgs& a, uint8_t* stg, int unit_u, int slot, int et) {
  const int kx = (unit_u % a.p.kb) * kTileK;
  const int r = et >> 3, ch = et & 7;
  const int tok = a.e.tok_base + r;
  if (a.xmode == X_FROM_H) {
    uint8_t* base = stg + slot * kStgFromHBytes;
    const float* src = a.xsrc + (long)tok * a.xsrc_ld + kx + ch * 8;
    cp_async16(base + (r * 64 + ch * 8) * 4, src);
    cp_async16(base + (r * 64 + ch * 8 + 4) * 4, src + 4);
    if (et < 16) cp_async16(base + 16 * 64 * 4 + et * 16, a.xgain + kx + et * 4);
  } else {
    uint8_t* base = stg + slot * kStgSwiBytes;
    const float* src = a.xsrc + (long)tok * a.xsrc_ld + (kx / 64) * 128 + ch * 8;
    cp_async16(base + (r * 64 + ch * 8) * 4, src);
    cp_async16(base + (r * 64 + ch * 8 + 4) * 4, src + 4);
    cp_async16(base + (16 * 64 + r * 64 + ch * 8) * 4, src + 64);
    cp_async16(base + (16 * 64 + r * 64 + ch * 8 + 4) * 4, src + 68);
    if (et < 16) cp_async4(base + 2 * 16 * 64 * 4 + et * 4, a.xrs + a.e.tok_base + et);
  }
  cp_async_commit();
}

// Convert the staged slot into the hi/lo operand planes of a stage.
__device__ __forceinline__ void stage_convert(const GemmArgs& a, const uint8_t* stg, int slot, uint8_t* xh,
                                              uint8_t* xl, int et) {
  const int r = et >> 3, ch = et & 7;
  float x[8];
  if (a.xmode == X_FROM_H) {
    const float* base = reinterpret_cast<const float*>(stg + slot * kStgFromHBytes);
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = base[r * 64 + ch * 8 + q] * base[16 * 64 + ch * 8 + q];
  } else {
    const float* base = reinterpret_cast<const float*>(stg + slot * kStgSwiBytes);
    const float rs = base[2 * 16 * 64 + r];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float gs = base[r * 64 + ch * 8 + q] * rs;
      x[q] = gs / (1.f + __expf(-gs)) * (base[16 * 64 + r * 64 + ch * 8 + q] * rs);
    }
  }
  if (r >= a.e.n_tok) {
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = 0.f;
  }
  uint4 hi, lo;
  split8(x, hi, lo);
  const int off = (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(xh + off) = hi;
  *reinterpret_cast<uint4*>(xl + off) = lo;
}

// Two CTAs fit per SM (registers <= 170, ~100 KB shared), so the next
// kernel's CTA can start its weight prefetch beside this one's tail.
__global__ void __launch_bounds__(kTcThreads, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, GemmArgs a,
                   TcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctl = smem + t.stages * t.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* empty = full + t.stages;
  uint64_t* xfull = empty + t.stages;
  uint64_t* accfull = xfull + t.stages;
  uint64_t* accempty = accfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort, last
  float* red = reinterpret_cast<float*>(ctl + 512);
  const bool xtma = a.xmode == X_PLANES;

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
      mbar_init(&xfull[s], kEpiThreads);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiThreads);
    }
    flags[0] = flags[1] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmW);
    if (xtma) tma_prefetch_map(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, t.tmem_cols);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 1, c0);   // 1: set-up done

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
      const uint32_t bytes = kWTileBytes + (xtma ? 2 * x_plane_bytes : 0u);
      auto load_x = [&](int i, int u) {
        if (!xtma) return;
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
      trace_mark(a.trace, blockIdx.x, 2, c0);               // 2: producer past the launch wait
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
          const uint32_t ph = (i / t.stages) & 1;
          if (!mbar_wait(&full[s], ph, &flags[0]) || (!xtma && !mbar_wait(&xfull[s], ph, &flags[0]))) {
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
      trace_mark(a.trace, blockIdx.x, 3, c0);                   // 3: last MMA issued
    }
  } else {
    // ------------------------------------------------------------------ converters + drain
    pdl_wait();
    const int et = threadIdx.x - 64;
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int row = 32 * q + lane;          // tile row (output feature) of this thread
    int conv = 0;                           // next unit whose operand planes to build
    // Build operand planes up to unit `upto` (exclusive), waiting for each
    // stage to be released by the MMA first.  A failed wait stops conversion
    // (the MMA then times out too) but keeps every barrier arrival.
    const bool staged = !xtma && t.nt == 16;     // cp.async pipeline (otherwise direct loads)
    const int D = staged ? stage_slots(a.xmode) : 0;
    uint8_t* stg = reinterpret_cast<uint8_t*>(red);   // the tile-epilogue scratch is unused here
    int issued = 0;
    auto convert_upto = [&](int upto) {
      if (xtma) return;
      for (; conv < upto; ++conv) {
        const int s = conv % t.stages;
        if (staged) {
          while (issued < n_units && issued < conv + D) {
            stage_issue(a, stg, u0 + issued, issued % D, et);
            ++issued;
          }
          cp_async_wait(issued - conv - 1);
          epi_sync();                    // every thread's copies of this unit have landed
        }
        bool got = true;
        if (conv >= t.stages) got = mbar_wait(&empty[s], ((conv / t.stages) & 1) ^ 1, &flags[0]);
        got = __all_sync(0xffffffffu, got);
        if (got) {
          uint8_t* st = smem + s * t.stage_bytes;
          if (staged) stage_convert(a, stg, conv % D, st + kWTileBytes, st + kWTileBytes + x_plane_bytes, et);
          else convert_unit(a, t, st + kWTileBytes, st + kWTileBytes + x_plane_bytes, ((u0 + conv) % p.kb) * kTileK,
                            et);
          fence_proxy_async_smem();
        } else {
          flags[0] = 1;
        }
        mbar_arrive(&xfull[s]);
        if (staged) epi_sync();          // the slot may be refilled only after everyone read it
      }
    };
    convert_upto(min(n_units, t.stages));
    // side duties, after the first stages are on their way
    if (a.rs_out && et < 32) {
      for (int tok = c; tok < a.e.n_tok; tok += p.grid) {
        const float* src = a.rs_src + (long)(a.e.tok_base + tok) * a.rs_ld;
        float ss = 0.f;
        for (int k = lane * 4; k < a.rs_len; k += 128) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + k));
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        if (lane == 0) a.rs_out[a.e.tok_base + tok] = rsqrtf(ss / (float)a.rs_len + a.e.g.eps);
      }
    }
    if (a.zero_ptr) {
      const long n4 = a.zero_n / 4;
      const long lo = n4 * c / p.grid, hi = n4 * (c + 1) / p.grid;
      for (long k = lo + et; k < hi; k += kEpiThreads)
        reinterpret_cast<float4*>(a.zero_ptr)[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int seg = 0, i_seg_end = 0;
    for (int u = u0; u < u1; ++seg) {
      const int T = u / p.kb;
      const int seg_end = min(u1, (T + 1) * p.kb);
      const int b = seg & 1, use = seg >> 1;
      const bool last_seg = seg_end == u1;
      i_seg_end += seg_end - u;
      convert_upto(min(n_units, i_seg_end + t.stages));
      // a failed wait skips the TMEM read but keeps every barrier arrival, so
      // no thread is left waiting at a named barrier
      const bool got = __all_sync(0xffffffffu, mbar_wait(&accfull[b], use & 1, &flags[0]));
      if (!got) flags[0] = 1;
      if (et == 0 && last_seg) trace_mark(a.trace, blockIdx.x, 6, c0);   // 6: last accumulator ready
      __syncwarp();
      tc_fence_after();
      if (a.omode == O_RED) {
        if (got) {
          float* dcol = a.dst + (long)a.e.tok_base * a.dst_ld + T * kTileN + row;
          const float wsc = a.e.wscale ? a.e.wscale[T * kTileN + row] : 1.f;
          for (int j0 = 0; j0 < a.e.n_tok; j0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * t.nt + j0), v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j0 + j < a.e.n_tok)
                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dcol + (long)(j0 + j) * a.dst_ld), "f"(v[j] * wsc)
                             : "memory");
          }
        }
        tc_fence_before();
        mbar_arrive(&accempty[b]);
      } else {
        float* acc_tile = a.acc + (long)T * kTileN * t.nt;
        if (got) {
          for (int j0 = 0; j0 < a.e.n_tok; j0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * t.nt + j0), v);
            acc_add16(acc_tile + (long)row * t.nt, j0, a.e.n_tok, v);
          }
        }
        tc_fence_before();
        mbar_arrive(&accempty[b]);
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
          if (et == 0) trace_mark(a.trace, blockIdx.x, last_seg ? 10 : 14, c0);   // 10/14: tile epilogue done
        }
      }
      u = seg_end;
    }
    if (et == 0) trace_mark(a.trace, blockIdx.x, 4, c0);        // 4: drain loop done
  }
  __syncwarp();   // role lanes rejoin their warp before the CTA barrier
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 5, c0);  // 5: all roles done
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

void launch_gemm_tc(const GemmArgs& a, const void* tmap_w, const void* tmap_x, cudaStream_t s) {
  TcCfg t{};
  t.nt = (a.e.n_tok + 15) / 16 * 16;
  t.stage_bytes = kWTileBytes + 2 * t.nt * 128;
  // ~100 KB per CTA lets the next kernel's CTA share the SM during the tail
  t.stages = std::max(2, std::min(8, (100 * 1024 - 512 - kRedFloats * 4) / t.stage_bytes));
  t.tmem_cols = pow2_at_least(2 * t.nt);
  t.x_row_lo = a.e.g.Mt;
  t.idesc = idesc_bf16(kTileN, t.nt);
  const size_t smem = gemm_tc_smem_bytes(t.nt, t.stages);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;   // the launch below is skipped; the caller's cudaGetLastError reports it
    attr_bytes = smem;
  }
  const CUtensorMap* mw = static_cast<const CUtensorMap*>(tmap_w);
  const CUtensorMap* mx = static_cast<const CUtensorMap*>(tmap_x ? tmap_x : tmap_w);
  launch_pdl(gemm_tc_kernel, dim3(a.p.grid), dim3(kTcThreads), smem, s, *mw, *mx, a, t);
}

}  // namespace dfl
