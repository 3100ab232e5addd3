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
      put_operand(f.op, idx + 0, f.op_plane, x.x, f.op_kind);
      put_operand(f.op, idx + 1, f.op_plane, x.y, f.op_kind);
      put_operand(f.op, idx + 2, f.op_plane, x.z, f.op_kind);
      put_operand(f.op, idx + 3, f.op_plane, x.w, f.op_kind);
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

// One warp per (token, head) row of the QKV accumulator.
template <int PER>
__device__ void qk_finish_row(const FinishArgs& f, int tok, int hh) {
  const Geo& g = f.g;
  constexpr int d = 32 * PER, half = d / 2;
  const int lane = threadIdx.x & 31, dim0 = lane * PER;
  const int kind = hh < g.Hq ? 0 : (hh < g.Hq + g.Hkv ? 1 : 2);
  const int head = kind == 0 ? hh : (kind == 1 ? hh - g.Hq : hh - g.Hq - g.Hkv);
  float* src = f.acc + (long)tok * g.qkv_n + hh * d + dim0;
  float x[PER], gn[PER];
  float2 cs[PER];
  if (PER == 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
    x[0] = v.x; x[1] = v.y;
  }
  const float* gsrc = kind == 0 ? f.qn : f.kn;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    gn[q] = kind != 2 ? gsrc[dim0 + q] : 1.f;
    cs[q] = kind != 2 ? f.rope_cs[(long)tok * half + (dim0 + q) % half] : make_float2(1.f, 0.f);
  }
  const int dst = kind != 0 ? f.dest[tok] : 0;
  // clear the accumulator row for the next layer
  if (PER == 4) *reinterpret_cast<float4*>(src) = make_float4(0.f, 0.f, 0.f, 0.f);
  else *reinterpret_cast<float2*>(src) = make_float2(0.f, 0.f);
  if (kind != 2) {
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < PER; ++q) ss += x[q] * x[q];
    ss = warp_sum(ss);
    const float rn = rsqrtf(ss / (float)d + g.eps);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const float y = x[q] * rn * gn[q];
      const float partner = __shfl_xor_sync(0xffffffffu, y, 16);   // dims j <-> j + d/2
      x[q] = lane < 16 ? (y * cs[q].x - partner * cs[q].y) : (y * cs[q].x + partner * cs[q].y);
    }
  }
  if (g.kvtype == KV_FP8 && kind == 0) {
    // an e4m3 cache stores K and V only: its queries stay f16
    __half* qrow = static_cast<__half*>(f.q_out) + ((long)tok * g.Hq + head) * d + dim0;
#pragma unroll
    for (int q = 0; q < PER; ++q) qrow[q] = __float2half_rn(x[q]);
  } else if (g.kvtype == KV_FP8) {
    put_row_fp8<PER>(g, x, lane, kind, f.layer, tok, head, dst, f.kpool, f.vpool);
  } else if (kind == 0) {
    const long base = ((long)tok * g.Hq + head) * d + dim0;
#pragma unroll
    for (int q = 0; q < PER; ++q) put_kv(f.q_out, base + q, x[q], g.kvtype);
  } else {
    const int page = dst >> 6, off = dst & (kPage - 1);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      if (kind == 1) put_kv(f.kpool, k_index(g, f.layer, page, head, off, dim0 + q), x[q], g.kvtype);
      else put_kv(f.vpool, v_index(g, f.layer, page, head, off, dim0 + q), x[q], g.kvtype);
    }
  }
}

__global__ void __launch_bounds__(128) qk_finish_kernel(FinishArgs f) {
  trace_cta_entry(f.trace);
  pdl_launch_dependents();
  pdl_wait();
  const Geo& g = f.g;
  const int heads = g.Hq + 2 * g.Hkv;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= f.n_tok * heads) return;
  const int tok = row / heads, hh = row % heads;
  if (g.d == 128) qk_finish_row<4>(f, tok, hh);
  else qk_finish_row<2>(f, tok, hh);
  trace_cta_exit(f.trace);
}

// One float4 of act per thread: a single round trip, no loop.
__global__ void __launch_bounds__(128) swiglu_kernel(FinishArgs f) {
  trace_cta_entry(f.trace);
  pdl_launch_dependents();
  pdl_wait();
  const Geo& g = f.g;
  const long n4 = (long)f.n_tok * g.I / 4;
  {
    const long k = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n4) {
      trace_cta_exit(f.trace);
      return;
    }
    const long e = k * 4;
    const int tok = (int)(e / g.I), j = (int)(e % g.I);
    float* gp = f.acc + (long)tok * 2 * g.I + (j / 64) * 128 + (j % 64);
    const float4 gv = __ldcg(reinterpret_cast<const float4*>(gp));
    const float4 uv = __ldcg(reinterpret_cast<const float4*>(gp + 64));
    *reinterpret_cast<float4*>(gp) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(gp + 64) = make_float4(0.f, 0.f, 0.f, 0.f);
    const float gg[4] = {gv.x, gv.y, gv.z, gv.w}, uu[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      put_operand(f.op, (long)tok * g.I + j + q, f.op_plane, gg[q] / (1.f + __expf(-gg[q])) * uu[q], f.op_kind);
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
    put_operand(op, idx + 0, plane, v.x, 0);
    put_operand(op, idx + 1, plane, v.y, 0);
    put_operand(op, idx + 2, plane, v.z, 0);
    put_operand(op, idx + 3, plane, v.w, 0);
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

int prep_norm_grid(const FinishArgs& f) { return f.n_tok; }

void launch_prep_norm(const FinishArgs& f, cudaStream_t s) {
  launch_pdl(prep_norm_kernel, dim3(prep_norm_grid(f)), dim3(kRowThreads), 0, s, f);
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

int qk_finish_grid(const FinishArgs& f) { return (f.n_tok * (f.g.Hq + 2 * f.g.Hkv) + 3) / 4; }

void launch_qk_finish(const FinishArgs& f, cudaStream_t s) {
  launch_pdl(qk_finish_kernel, dim3(qk_finish_grid(f)), dim3(128), 0, s, f);
}

int swiglu_grid(const FinishArgs& f, int n_sm) {
  (void)n_sm;
  const long n4 = (long)f.n_tok * f.g.I / 4;
  return (int)((n4 + 127) / 128);
}

void launch_swiglu(const FinishArgs& f, int n_sm, cudaStream_t s) {
  launch_pdl(swiglu_kernel, dim3(swiglu_grid(f, n_sm)), dim3(128), 0, s, f);
}

}  // namespace dfl
