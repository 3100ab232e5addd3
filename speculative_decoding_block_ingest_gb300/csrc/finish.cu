// finish.cu -- the small element-wise steps between the round's projections.
//
// They run as short, wide kernels between the weight-streaming ones (chained
// by programmatic dependent launch) so that no latency-bound step sits inside
// a kernel that streams HBM at full rate:
//   final_norm   the round's closing RMSNorm into the f32 output rows;
//   prep_norm    RMSNorm operand of the next projection: per token row,
//                x = h * gain * rsqrt(mean(h^2) + eps) as hi/lo bf16 planes
//                (or f32 for f32 drafters);
//   qk_finish    per (token, head) row of the QKV accumulator: q and k head
//                RMSNorm + NeoX RoPE (mscale folded into the table); q to the
//                attention's query buffer, the block rows' K and V into the
//                KV pages (rows len .. len+15, transient); the row is cleared;
//   swiglu       act = silu(g) * u from the gate/up accumulator as hi/lo
//                planes; the entries are cleared.
#include <algorithm>
#include <cmath>

#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

// Row kernels: one CTA of kRowThreads per token row, every load of the row
// (and of the gain) issued before the first use, so a row costs one L2 round
// trip plus a block reduction.
constexpr int kRowThreads = 256;
constexpr int kRowVec = kMaxHidden / (4 * kRowThreads);   // float4 per thread

__device__ __forceinline__ float block_sum_rows(float v) {
  __shared__ float red[kRowThreads / 32];
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += red[w];
  return t;
}

// x = row * gain * rsqrt(mean(row^2) + eps) for the row's float4 slots this
// thread owns (slot tid + k * kRowThreads); returns false for unused slots.
struct RowNorm {
  float4 v[kRowVec], w[kRowVec];
  float r;
  __device__ void load(const float* row, const float* gain, int H, float eps) {
    const int n4 = H / 4;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const float4* g4 = reinterpret_cast<const float4*>(gain);
#pragma unroll
    for (int k = 0; k < kRowVec; ++k) {
      const int i = threadIdx.x + k * kRowThreads;
      v[k] = i < n4 ? __ldcg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      w[k] = i < n4 ? __ldg(g4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kRowVec; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    r = rsqrtf(block_sum_rows(ss) / (float)H + eps);
  }
  __device__ float4 out(int k) const {
    return make_float4(v[k].x * w[k].x * r, v[k].y * w[k].y * r, v[k].z * w[k].z * r, v[k].w * w[k].w * r);
  }
};

__global__ void __launch_bounds__(kRowThreads) prep_norm_kernel(FinishArgs f) {
  trace_cta_entry(f.trace);
  pdl_launch_dependents();
  pdl_wait();
  const int tok = blockIdx.x;
  const Geo& g = f.g;
  RowNorm rn;
  rn.load(f.h + (long)tok * g.H, f.gain, g.H, g.eps);
#pragma unroll
  for (int k = 0; k < kRowVec; ++k) {
    const int i = threadIdx.x + k * kRowThreads;
    if (4 * i < g.H) {
      const float4 x = rn.out(k);
      const long idx = (long)tok * g.H + 4 * i;
      if (f.u_out) reinterpret_cast<float4*>(f.u_out + idx)[0] = x;
      put_operand4(f.op, idx, f.op_plane, x, f.op_kind);
    }
  }
  trace_cta_exit(f.trace);
}

// Wide passes (more than 64 rows): one warp per token row, the row's VEC
// float4 per lane (and the gain's) loaded at once and the sum of squares
// taken by warp shuffles; a CTA of kRowWarps rows, so a pass of 512 rows is
// 128 CTAs instead of 512.
constexpr int kRowWarps = 4;
template <int VEC>
__global__ void __launch_bounds__(32 * kRowWarps) prep_norm_warp_kernel(FinishArgs f) {
  trace_cta_entry(f.trace);
  pdl_launch_dependents();
  pdl_wait();
  const Geo& g = f.g;
  const int lane = threadIdx.x & 31;
  const int tok = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (tok < f.n_tok) {
    const float4* r4 = reinterpret_cast<const float4*>(f.h + (long)tok * g.H);
    const float4* g4 = reinterpret_cast<const float4*>(f.gain);
    float4 v[VEC], w[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      v[k] = __ldcg(r4 + lane + 32 * k);
      w[k] = __ldg(g4 + lane + 32 * k);
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VEC; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    const float r = rsqrtf(warp_sum(ss) / (float)g.H + g.eps);
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const float4 x = make_float4(v[k].x * w[k].x * r, v[k].y * w[k].y * r, v[k].z * w[k].z * r, v[k].w * w[k].w * r);
      const long idx = (long)tok * g.H + 4 * (lane + 32 * k);
      if (f.u_out) reinterpret_cast<float4*>(f.u_out + idx)[0] = x;
      put_operand4(f.op, idx, f.op_plane, x, f.op_kind);
    }
  }
  trace_cta_exit(f.trace);
}

// Final RMSNorm of the residual stream into the f32 output rows.
__global__ void __launch_bounds__(kRowThreads) final_norm_kernel(const float* h, const float* gain, float* out, int H,
                                                               float eps, unsigned long long* trace) {
  trace_cta_entry(trace);
  pdl_launch_dependents();
  pdl_wait();
  const int tok = blockIdx.x;
  RowNorm rn;
  rn.load(h + (long)tok * H, gain, H, eps);
  float4* o4 = reinterpret_cast<float4*>(out + (long)tok * H);
#pragma unroll
  for (int k = 0; k < kRowVec; ++k) {
    const int i = threadIdx.x + k * kRowThreads;
    if (4 * i < H) o4[i] = rn.out(k);
  }
  trace_cta_exit(trace);
}

// One warp per (token, head) row of the QKV accumulator, RPW rows per warp
// (rows w, w + W, ... for W warps in the grid): the accumulator and RoPE
// loads of all of a warp's rows are issued before the first row is
// finished (its stores may alias later rows, so the compiler would not
// hoist them).
template <int PER, int RPW>
__device__ void qk_finish_rows(const FinishArgs& f, int row0, int rstride) {
  const Geo& g = f.g;
  constexpr int d = 32 * PER, half = d / 2;
  const int heads = g.Hq + 2 * g.Hkv, n_rows = f.n_tok * heads;
  const int lane = threadIdx.x & 31, dim0 = lane * PER;
  float x[RPW][PER];
  float2 cs[RPW][PER];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = row0 + r * rstride;
    if (row >= n_rows) break;
    const int tok = row / heads, hh = row % heads;
    const float* src = f.acc + (long)tok * g.qkv_n + hh * d + dim0;
    if (PER == 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
      x[r][0] = v.x; x[r][1] = v.y; x[r][2] = v.z; x[r][3] = v.w;
    } else {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
      x[r][0] = v.x; x[r][1] = v.y;
    }
    const bool roped = hh < g.Hq + g.Hkv;
#pragma unroll
    for (int q = 0; q < PER; ++q)
      cs[r][q] = roped ? f.rope_cs[(long)tok * half + (dim0 + q) % half] : make_float2(1.f, 0.f);
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = row0 + r * rstride;
    if (row >= n_rows) break;
    const int tok = row / heads, hh = row % heads;
    const int kind = hh < g.Hq ? 0 : (hh < g.Hq + g.Hkv ? 1 : 2);
    const int head = kind == 0 ? hh : (kind == 1 ? hh - g.Hq : hh - g.Hq - g.Hkv);
    float* src = f.acc + (long)tok * g.qkv_n + hh * d + dim0;
    // clear the accumulator row for the next layer
    if (PER == 4) *reinterpret_cast<float4*>(src) = make_float4(0.f, 0.f, 0.f, 0.f);
    else *reinterpret_cast<float2*>(src) = make_float2(0.f, 0.f);
    float* xr = x[r];
    if (kind != 2) {
      const float* gsrc = kind == 0 ? f.qn : f.kn;
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < PER; ++q) ss += xr[q] * xr[q];
      ss = warp_sum(ss);
      const float rn = rsqrtf(ss / (float)d + g.eps);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const float y = xr[q] * rn * gsrc[dim0 + q];
        const float partner = __shfl_xor_sync(0xffffffffu, y, 16);   // dims j <-> j + d/2
        xr[q] = lane < 16 ? (y * cs[r][q].x - partner * cs[r][q].y) : (y * cs[r][q].x + partner * cs[r][q].y);
      }
    }
    const int dst = kind != 0 ? f.dest[tok] : 0;
    if (g.kvtype == KV_FP8 && kind == 0) {
      // an e4m3 cache stores K and V only: its queries stay f16
      __half* qrow = static_cast<__half*>(f.q_out) + ((long)tok * g.Hq + head) * d + dim0;
#pragma unroll
      for (int q = 0; q < PER; ++q) qrow[q] = __float2half_rn(xr[q]);
    } else if (g.kvtype == KV_FP8) {
      put_row_fp8<PER>(g, xr, lane, kind, f.layer, tok, head, dst, f.kpool, f.vpool);
    } else if (kind == 0) {
      put_kv_row<PER>(f.q_out, ((long)tok * g.Hq + head) * d + dim0, xr, g.kvtype);
    } else {
      const int page = dst >> 6, off = dst & (kPage - 1);
      if (kind == 1) {
        put_kv_row<PER>(f.kpool, k_index(g, f.layer, page, head, off, dim0), xr, g.kvtype);
      } else {
#pragma unroll
        for (int q = 0; q < PER; ++q) put_kv(f.vpool, v_index(g, f.layer, page, head, off, dim0 + q), xr[q], g.kvtype);
      }
    }
  }
}

template <int RPW>
__global__ void __launch_bounds__(256) qk_finish_kernel(FinishArgs f) {
  trace_cta_entry(f.trace);
  pdl_launch_dependents();
  pdl_wait();
  const int wpc = blockDim.x >> 5;
  const int row0 = blockIdx.x * wpc + (threadIdx.x >> 5), rstride = gridDim.x * wpc;
  if (f.g.d == 128) qk_finish_rows<4, RPW>(f, row0, rstride);
  else qk_finish_rows<2, RPW>(f, row0, rstride);
  trace_cta_exit(f.trace);
}

// Four float4 of act per thread per pass, every gate and up load of a pass
// issued before the first store (the stores may alias later loads, so the
// compiler would not hoist them), over a grid of at most two CTAs per SM.
constexpr int kSwiThreads = 256;
constexpr int kSwiVec = 4;
__global__ void __launch_bounds__(kSwiThreads) swiglu_kernel(FinishArgs f) {
  trace_cta_entry(f.trace);
  pdl_launch_dependents();
  pdl_wait();
  const Geo& g = f.g;
  const long n4 = (long)f.n_tok * g.I / 4;
  const long stride = (long)gridDim.x * kSwiThreads;
  for (long k0 = (long)blockIdx.x * kSwiThreads + threadIdx.x; k0 < n4; k0 += kSwiVec * stride) {
    float4 gv[kSwiVec], uv[kSwiVec];
#pragma unroll
    for (int q = 0; q < kSwiVec; ++q) {
      const long k = k0 + q * stride;
      if (k < n4) {
        const long e = k * 4;
        const float* gp = f.acc + (e / g.I) * 2 * g.I + ((e % g.I) / 64) * 128 + (e % 64);
        gv[q] = __ldcg(reinterpret_cast<const float4*>(gp));
        uv[q] = __ldcg(reinterpret_cast<const float4*>(gp + 64));
      }
    }
#pragma unroll
    for (int q = 0; q < kSwiVec; ++q) {
      const long k = k0 + q * stride;
      if (k < n4) {
        const long e = k * 4;
        const int tok = (int)(e / g.I), j = (int)(e % g.I);
        float* gp = f.acc + (long)tok * 2 * g.I + (j / 64) * 128 + (j % 64);
        *reinterpret_cast<float4*>(gp) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(gp + 64) = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 a = make_float4(gv[q].x / (1.f + __expf(-gv[q].x)) * uv[q].x,
                                     gv[q].y / (1.f + __expf(-gv[q].y)) * uv[q].y,
                                     gv[q].z / (1.f + __expf(-gv[q].z)) * uv[q].z,
                                     gv[q].w / (1.f + __expf(-gv[q].w)) * uv[q].w);
        put_operand4(f.op, (long)tok * g.I + j, f.op_plane, a, f.op_kind);
      }
    }
  }
  trace_cta_exit(f.trace);
}

// f32 rows -> hi/lo bf16 operand planes (no norm): the lm_head's operand.
__global__ void __launch_bounds__(kRowThreads) to_operand_kernel(const float* src, int width, void* op, long plane) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x, n4 = width / 4;
  const float4* r4 = reinterpret_cast<const float4*>(src + (long)row * width);
  for (int c = threadIdx.x; c < n4; c += kRowThreads) {
    const float4 v = __ldg(r4 + c);
    const long idx = (long)row * width + 4 * c;
    put_operand4(op, idx, plane, v, OPK_BF16);
  }
}

// Row argmax over `V` logits, lowest index among equal maxima.
__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(kRowThreads) argmax_kernel(const float* logits, int V, int32_t* tokens) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const float4* l4 = reinterpret_cast<const float4*>(logits + (long)row * V);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  // each thread walks its float4s in increasing index order
  for (int c = threadIdx.x; c < V / 4; c += kRowThreads) {
    const float4 v = __ldcg(l4 + c);
    better(bv, bi, v.x, 4 * c);
    better(bv, bi, v.y, 4 * c + 1);
    better(bv, bi, v.z, 4 * c + 2);
    better(bv, bi, v.w, 4 * c + 3);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  __shared__ float sv[kRowThreads / 32];
  __shared__ int si[kRowThreads / 32];
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = bv;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kRowThreads / 32; ++w) better(bv, bi, sv[w], si[w]);
    tokens[row] = bi;
  }
}

void launch_to_operand(const float* src, int n_rows, int width, void* op, long plane, cudaStream_t s) {
  launch_pdl(to_operand_kernel, dim3(n_rows), dim3(kRowThreads), 0, s, src, width, op, plane);
}

void launch_argmax(const float* logits, int n_rows, int V, int32_t* tokens, cudaStream_t s) {
  launch_pdl(argmax_kernel, dim3(n_rows), dim3(kRowThreads), 0, s, logits, V, tokens);
}

// float4 per lane of the warp-per-row form (a row of 1024 or 2048), else 0
static int prep_norm_vec(const FinishArgs& f) {
  if (f.n_tok <= 64 || f.g.H % 128) return 0;
  const int vec = f.g.H / 128;
  return (vec == 8 || vec == 16) ? vec : 0;
}

int prep_norm_grid(const FinishArgs& f) {
  return prep_norm_vec(f) ? (f.n_tok + kRowWarps - 1) / kRowWarps : f.n_tok;
}

void launch_prep_norm(const FinishArgs& f, cudaStream_t s) {
  const dim3 grid(prep_norm_grid(f)), warps(32 * kRowWarps);
  switch (prep_norm_vec(f)) {
    case 8: launch_pdl(prep_norm_warp_kernel<8>, grid, warps, 0, s, f); break;
    case 16: launch_pdl(prep_norm_warp_kernel<16>, grid, warps, 0, s, f); break;
    default: launch_pdl(prep_norm_kernel, grid, dim3(kRowThreads), 0, s, f);
  }
}

const void* final_norm_kernel_entry() { return reinterpret_cast<const void*>(final_norm_kernel); }

void launch_final_norm(const float* h, const float* gain, float* out, int n_tok, const Geo& g,
                       unsigned long long* trace, cudaStream_t s) {
  launch_pdl(final_norm_kernel, dim3(n_tok), dim3(kRowThreads), 0, s, h, gain, out, g.H, g.eps, trace);
}

// DFlash2 conv (memra_engine::dflash, Dflash2Conv; DflashDraft, d2_conv_prepare / d2_conv_finish):
// out_t[c] = (base[half][c][0] + dyn_t[half][g][0]) * src_{t-1}[c]
//          + (base[half][c][1] + dyn_t[half][g][1]) * src_t[c],  g = c / (H / groups),
// src_{t-1} = 0 for the first block row of a sequence.  Four channels per
// thread; prepare writes the operand planes (and clears the next
// projections' red.add targets), finish adds into the residual stream.
__global__ void __launch_bounds__(256) conv_kernel(ConvArgs a) {
  trace_cta_entry(a.trace);
  pdl_launch_dependents();
  pdl_wait();
  const Geo& g = a.g;
  const long stride = (long)gridDim.x * blockDim.x;
  const long t0 = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (a.half == 0) {
    for (long i = t0; i < a.zero0_n; i += stride) a.zero0[i] = 0.f;
    for (long i = t0; i < a.zero1_n; i += stride) a.zero1[i] = 0.f;
  }
  const int n4 = g.H / 4, gs = g.H / a.groups;
  const float* b = a.base + (long)a.half * g.H * 2;
  for (long e = t0; e < (long)a.n_tok * n4; e += stride) {
    const int t = (int)(e / n4), c = (int)(e % n4) * 4;
    const float4 cur = __ldcg(reinterpret_cast<const float4*>(a.src + (long)t * g.H + c));
    const float4 prv = (t % kBlock) ? __ldcg(reinterpret_cast<const float4*>(a.src + (long)(t - 1) * g.H + c))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
    const float* dy = a.dyn + (long)t * a.dyn_ld + (long)a.half * a.groups * 2;
    const float xc[4] = {cur.x, cur.y, cur.z, cur.w}, xp[4] = {prv.x, prv.y, prv.z, prv.w};
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ch = c + j, grp = ch / gs;
      o[j] = (b[2 * ch] + dy[2 * grp]) * xp[j] + (b[2 * ch + 1] + dy[2 * grp + 1]) * xc[j];
    }
    const long idx = (long)t * g.H + c;
    if (a.half == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) put_operand(a.op, idx + j, a.op_plane, o[j], a.op_kind);
    } else {
      float4* hp = reinterpret_cast<float4*>(a.h + idx);
      const float4 hv = *hp;
      *hp = make_float4(hv.x + o[0], hv.y + o[1], hv.z + o[2], hv.w + o[3]);
    }
  }
  trace_cta_exit(a.trace);
}

int conv_grid(const ConvArgs& c, int n_sm) {
  const long n = std::max<long>((long)c.n_tok * c.g.H / 4, std::max(c.zero0_n, c.zero1_n));
  return (int)std::max<long>(1, std::min<long>((n + 255) / 256, 4L * n_sm));
}

void launch_conv(const ConvArgs& c, int n_sm, cudaStream_t s) {
  launch_pdl(conv_kernel, dim3(conv_grid(c, n_sm)), dim3(256), 0, s, c);
}

// Rows per warp (2 at d = 128 once a pass has more rows than about eight
// warps per SM, else 1) and warps per CTA (4 for one row a warp, else 8).
// Four rows a warp (half the CTAs again) was 1% slower at 32 sequences.
static void qk_finish_shape(const FinishArgs& f, int n_sm, int* rpw, int* wpc) {
  const long rows = (long)f.n_tok * (f.g.Hq + 2 * f.g.Hkv);
  *rpw = f.g.d == 128 && rows > 8L * n_sm ? 2 : 1;
  *wpc = *rpw == 1 ? 4 : 8;
}

int qk_finish_grid(const FinishArgs& f, int n_sm) {
  int rpw, wpc;
  qk_finish_shape(f, n_sm, &rpw, &wpc);
  const long rows = (long)f.n_tok * (f.g.Hq + 2 * f.g.Hkv);
  return (int)((rows + (long)rpw * wpc - 1) / ((long)rpw * wpc));
}

void launch_qk_finish(const FinishArgs& f, int n_sm, cudaStream_t s) {
  int rpw, wpc;
  qk_finish_shape(f, n_sm, &rpw, &wpc);
  const dim3 grid(qk_finish_grid(f, n_sm)), block(32 * wpc);
  if (rpw == 1) launch_pdl(qk_finish_kernel<1>, grid, block, 0, s, f);
  else launch_pdl(qk_finish_kernel<2>, grid, block, 0, s, f);
}

int swiglu_grid(const FinishArgs& f, int n_sm) {
  const long n4 = (long)f.n_tok * f.g.I / 4;
  const long per_cta = (long)kSwiThreads * kSwiVec;
  return (int)std::max<long>(1, std::min<long>((n4 + per_cta - 1) / per_cta, 2L * n_sm));
}

void launch_swiglu(const FinishArgs& f, int n_sm, cudaStream_t s) {
  launch_pdl(swiglu_kernel, dim3(swiglu_grid(f, n_sm)), dim3(kSwiThreads), 0, s, f);
}

}  // namespace dfl
