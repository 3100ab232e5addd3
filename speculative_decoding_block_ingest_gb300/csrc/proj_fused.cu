// proj_fused.cu -- a projection that owns whole output tiles, with its
// RMSNorm operand built in the kernel and its element-wise step fused into
// the epilogue.
//
// One CTA per 128-row weight tile, over the full K (no stream-K split), so a
// tile's result is complete in the CTA's TMEM and the step after the
// projection needs no further launch and no accumulator round trip through
// L2.  The operand is RMSNorm(h) with the norm's gain: the CTA multiplies
// h by the gain as it goes and applies rsqrt(mean(h^2) + eps) to the finished
// outputs (the projection is linear, so the row scale commutes with it),
// where mean(h^2) comes from the h values the CTA has read anyway (it reads
// the whole row: every K column belongs to its tile).  Epilogues:
//   gate/up  rows 0..63 of tile T are gate rows 64T.., rows 64..127 the
//            matching up rows; act[tok][64T + j] = silu(g_j) * u_j into the
//            down projection's hi/lo bf16 operand planes (the DflashDraft
//            forward_round MLP: SiLU-gated, post-attention RMSNorm input).
// Warps (7 x 32 threads):
//   0 (one lane)  producer: the tile's 16 KB weight blocks (bulk copies; the
//                 first stages before the programmatic-launch wait) and, after
//                 the wait, the matching [nt x 64] f32 slices of h (TMA);
//   1, 2 (one lane each)  MMA issuers: unit kb goes to issuer kb % 2, each
//                 accumulating into its own TMEM accumulator (two issuers
//                 overlap the tensor core's per-instruction latency);
//   3..6          converters: per unit, h slice x gain -> hi/lo bf16 operand
//                 rows in the 128-byte swizzle, and the rows' sums of
//                 squares; then the epilogue.
#include <algorithm>
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kOwnThreads = 224;
constexpr int kOwnCvTid0 = 96;          // first converter thread (warp 3)
constexpr int kOwnCv = 128;
constexpr int kOwnBar = 2;              // named barrier of the converter warps
constexpr int kWBlk = kTileN * kTileK * 2;   // 16 KB

struct OwnCfg {
  int nt;            // token columns (16 or 32)
  int stages;        // even: stage kb % stages belongs to issuer kb % 2
  int stage_bytes;   // weights + operand hi/lo (2 x nt x 128 B) + h slice (nt x 256 B)
  int aw;            // accumulator columns (2 nt: hi and lo in one MMA)
  uint32_t idesc;
};

__device__ __forceinline__ void own_sync() {
  asm volatile("barrier.sync %0, %1;" ::"r"(kOwnBar), "r"(kOwnCv) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace

__global__ void __launch_bounds__(kOwnThreads, 1)
    proj_own_kernel(const __grid_constant__ CUtensorMap tmH, OwnArgs a, OwnCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctl = smem + t.stages * t.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);     // [stages] weights + h slice landed
  uint64_t* opready = full + t.stages;                   // [stages] operand converted
  uint64_t* empty = opready + t.stages;                  // [stages] MMAs of the stage done
  uint64_t* accfull = empty + t.stages;                  // [2] issuer's accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 2);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort
  float* red = reinterpret_cast<float*>(ctl + 512);      // [128][nt + 1] finished tile
  float* rsc = red + kTileN * (t.nt + 1);                // [nt] row scales
  float* sgain = rsc + 32;                               // [K] the norm's gain

  const Geo& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = blockIdx.x;                              // this CTA's tile
  const int nkb = a.kb;
  const uint32_t plane = (uint32_t)t.nt * 128;           // one operand plane of a stage
  const uint32_t hbytes = (uint32_t)t.nt * kTileK * 4;   // one h slice
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
      mbar_init(&opready[s], kOwnCv);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&accfull[0], 1);
    mbar_init(&accfull[1], 1);
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmH);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 2 * t.aw < 32 ? 32 : 2 * t.aw);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 1, c0);   // 1: set-up done

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      const uint64_t pol = policy_evict_first();
      const uint8_t* wsrc = a.W + (size_t)T * nkb * kWBlk;
      const uint32_t bytes = kWBlk + hbytes;
      const int pre = min(nkb, t.stages);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], bytes);
        bulk_load_hint(smem + i * t.stage_bytes, wsrc + (size_t)i * kWBlk, kWBlk, &full[i], pol);
      }
      // h is the residual stream the predecessor finished
      pdl_wait();
      pdl_launch_dependents();
      trace_mark(a.trace, blockIdx.x, 2, c0);                 // 2: producer past the launch wait
      const uint32_t hoff = kWBlk + 2 * plane;
      for (int i = 0; i < pre; ++i) tma_load_2d(smem + i * t.stage_bytes + hoff, &tmH, &full[i], i * kTileK, 0);
      int st = 0;
      uint32_t ph = 0;
      for (int i = pre; i < nkb; ++i) {
        if (!mbar_wait(&empty[st], ph, &flags[0])) {
          flags[0] = 1;
          break;
        }
        uint8_t* sp = smem + st * t.stage_bytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_load_hint(sp, wsrc + (size_t)i * kWBlk, kWBlk, &full[st], pol);
        tma_load_2d(sp + hoff, &tmH, &full[st], i * kTileK, 0);
        if (++st == t.stages) {
          st = 0;
          ph ^= 1;
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuers
      const int j = warp - 1;
      const uint64_t d0 = desc_sw128(smem_u32(smem));
      const uint32_t dstage = (uint32_t)t.stage_bytes >> 4;
      constexpr uint32_t xo = kWBlk >> 4;
      const uint32_t acc = tmem + (uint32_t)(j * t.aw);
      int st = j;
      uint32_t ph = 0;
      bool ok = true;
      int k = 0;
      for (int kb = j; kb < nkb; kb += 2, ++k) {
        if (!mbar_wait(&full[st], ph, &flags[0]) || !mbar_wait(&opready[st], ph, &flags[0])) {
          flags[0] = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dw = d0 + (uint64_t)(st * dstage);
#pragma unroll
        for (uint32_t kk = 0; kk < 8; kk += 2) mma_bf16(acc, dw + kk, dw + xo + kk, t.idesc, (k > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&empty[st]);
        st += 2;
        if (st >= t.stages) {
          st -= t.stages;
          ph ^= 1;
        }
      }
      // committed also after a failure: the drain's wait ends either way
      mma_commit(&accfull[j]);
      (void)ok;
      if (j == 0) trace_mark(a.trace, blockIdx.x, 3, c0);       // 3: last MMA issued
    }
  } else {
    // ------------------------------------------------------------------ converters, then the epilogue
    pdl_wait();
    const int ct = threadIdx.x - kOwnCvTid0;   // 0..127
    const int c8 = ct & 7;                     // 8-column piece of a 64-column slice
    const int t0 = ct >> 3;                    // token (and t0 + 16 when nt = 32)
    const int ntp = t.nt / 16;                 // tokens per thread
    // the gain once into shared memory (a global load per unit would put an
    // L2 round trip on every unit's critical path)
    for (int i = ct; i < nkb * kTileK / 4; i += kOwnCv)
      reinterpret_cast<float4*>(sgain)[i] = __ldg(reinterpret_cast<const float4*>(a.gain) + i);
    own_sync();
    float ss[2] = {0.f, 0.f};
    bool ok = true;
    int st = 0;
    uint32_t ph = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const float4* gsrc = reinterpret_cast<const float4*>(sgain + kb * kTileK + c8 * 8);
      const float4 g0 = gsrc[0], g1 = gsrc[1];
      const bool got = __all_sync(0xffffffffu, ok && mbar_wait(&full[st], ph, &flags[0]));
      if (!got) ok = false;
      __syncwarp();
      uint8_t* sp = smem + st * t.stage_bytes;
      if (ok) {
        const float* hs = reinterpret_cast<const float*>(sp + kWBlk + 2 * plane);
        for (int q = 0; q < ntp; ++q) {
          const int tok = t0 + 16 * q;
          const float4 x0 = *reinterpret_cast<const float4*>(hs + tok * kTileK + c8 * 8);
          const float4 x1 = *reinterpret_cast<const float4*>(hs + tok * kTileK + c8 * 8 + 4);
          const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          const float gn[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            ss[q] += x[e] * x[e] + x[e + 1] * x[e + 1];
            const float y0 = x[e] * gn[e], y1 = x[e + 1] * gn[e + 1];
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(y0, y1);
            const float2 hf = __bfloat1622float2(h2);
            hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            lo[e / 2] = pack_bf16x2(y0 - hf.x, y1 - hf.y);
          }
          const uint32_t off = (uint32_t)tok * 128 + (uint32_t)((c8 ^ (tok & 7)) << 4);
          *reinterpret_cast<uint4*>(sp + kWBlk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sp + kWBlk + plane + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&opready[st]);
      if (++st == t.stages) {
        st = 0;
        ph ^= 1;
      }
    }
    // row scales: the 8 threads of a token (consecutive lanes) add their sums
    for (int q = 0; q < ntp; ++q) {
      float v = ss[q];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      if (c8 == 0) rsc[t0 + 16 * q] = rsqrtf(v / (float)(nkb * kTileK) + g.eps);
    }
    // the finished tile: row f = this thread's TMEM lane, both issuers, hi + lo
    const int qd = warp & 3;
    const int f = 32 * qd + lane;
    bool got = true;
    for (int jj = 0; jj < 2; ++jj) got = __all_sync(0xffffffffu, mbar_wait(&accfull[jj], 0, &flags[0])) && got;
    if (!got) ok = false;
    __syncwarp();
    tc_fence_after();
    if (ok) {
      const float wsc = a.wscale ? a.wscale[T * kTileN + f] : 1.f;
      for (int j0 = 0; j0 < t.nt; j0 += 16) {
        float v[16] = {};
        for (int jj = 0; jj < 2; ++jj) {
          if (jj >= nkb) break;   // an issuer without units left its accumulator unwritten
          float w[16];
          const uint32_t base = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(jj * t.aw + j0);
          tmem_ld16(base, w);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] += w[e];
          tmem_ld16(base + (uint32_t)t.nt, w);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] += w[e];
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) red[f * (t.nt + 1) + j0 + e] = v[e] * wsc;
      }
    }
    tc_fence_before();
    own_sync();
    if (ok && a.epi == OWN_SWIGLU) {
      // act[tok][64 T + jc] = silu(r g) * (r u); thread: column jc, tokens
      // ct / 64, + 2, ...
      const int jc = ct & 63;
      for (int tok = ct >> 6; tok < a.n_tok; tok += 2) {
        const float r = rsc[tok];
        const float gv = red[jc * (t.nt + 1) + tok] * r;
        const float uv = red[(64 + jc) * (t.nt + 1) + tok] * r;
        put_operand(a.out, (long)tok * a.out_ld + T * 64 + jc, a.out_plane, gv / (1.f + __expf(-gv)) * uv, 0);
      }
    }
    if (ct == 0) trace_mark(a.trace, blockIdx.x, 4, c0);   // 4: epilogue done
  }
  __syncwarp();
  __syncthreads();
  trace_exit_warp(a.trace, blockIdx.x);
  if (flags[0] && threadIdx.x == 0) atomicExch(a.err, DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 2 * t.aw < 32 ? 32 : 2 * t.aw);
  }
}

size_t proj_own_smem_bytes(int nt, int stages, int K) {
  const int stage_bytes = kWBlk + nt * 512;
  return (size_t)stages * stage_bytes + 512 + (size_t)(kTileN * (nt + 1) + 32 + K) * 4 + 1024;
}

cudaError_t launch_proj_own(const OwnArgs& a, const void* tmap_h, cudaStream_t s) {
  OwnCfg t{};
  t.nt = (a.n_tok + 15) / 16 * 16;
  if (t.nt > 32) return cudaErrorInvalidValue;
  t.stage_bytes = kWBlk + t.nt * 512;
  t.stages = 12;
  const int K = a.kb * kTileK;
  while (t.stages > 2 && proj_own_smem_bytes(t.nt, t.stages, K) > 227u * 1024u) t.stages -= 2;
  t.aw = 2 * t.nt;
  t.idesc = idesc_bf16(kTileN, t.aw);
  const size_t smem = proj_own_smem_bytes(t.nt, t.stages, K);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    const cudaError_t e = cudaFuncSetAttribute(proj_own_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_bytes = smem;
  }
  return launch_pdl(proj_own_kernel, dim3(a.n_tiles), dim3(kOwnThreads), smem, s,
                    *static_cast<const CUtensorMap*>(tmap_h), a, t);
}

}  // namespace dfl
