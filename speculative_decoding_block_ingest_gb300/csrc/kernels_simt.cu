// kernels_simt.cu -- CUDA-core kernels of the drafter round.
//
//  * gemm_simt: the f32-weight projection (f32 drafters need FFMA accuracy;
//    TF32 tensor math would not meet their tolerance), same stream-K split
//    and shared epilogue as the tensor-core projection;
//  * attention over the paged KV cache for f32 caches, and the split-KV
//    combine used by every attention path;
//  * the per-call init kernels (descriptor upload, page-table update,
//    residual stream / operand set-up), the final norm and KV read-back.
#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

// ------------------------------------------------------------------ GEMM (CUDA cores)
__device__ __forceinline__ float load_w(const void* W, long idx, int wtype) {
  if (wtype == W_F32) return __ldg(reinterpret_cast<const float*>(W) + idx);
  if (wtype == W_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(W)[idx]);
  __nv_fp8_e4m3 v;
  v.__x = reinterpret_cast<const __nv_fp8_storage_t*>(W)[idx];
  return float(v);
}

__device__ __forceinline__ float load_x(const GemmArgs& a, int tok, int k) {
  const long idx = (long)tok * a.x_ld + k;
  if (a.x_f32) return reinterpret_cast<const float*>(a.X)[idx];
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(a.X);
  return __bfloat162float(x[idx]) + __bfloat162float(x[idx + a.x_plane]);
}

constexpr int kSimtTok = 16;

__global__ void __launch_bounds__(128) gemm_simt_kernel(GemmArgs a) {
  __shared__ float smem[kTileN * (kTileK + 1) + kSimtTok * kTileK];
  __shared__ int s_last;
  float* Ws = smem;                          // [128][65]
  float* Xs = smem + kTileN * (kTileK + 1);  // [16][64]
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const Part p = a.p;
  const int u1 = p.start(c + 1);
  const int nt = (a.e.n_tok + 15) / 16 * 16;
  for (int u = p.start(c); u < u1;) {
    const int T = u / p.kb;
    const int seg_end = min(u1, (T + 1) * p.kb);
    const int kb0 = u - T * p.kb, kb1 = seg_end - T * p.kb;
    float* acc_tile = a.acc + (long)T * kTileN * nt;
    for (int tok0 = 0; tok0 < a.e.n_tok; tok0 += kSimtTok) {
      float acc[kSimtTok];
#pragma unroll
      for (int t = 0; t < kSimtTok; ++t) acc[t] = 0.f;
      for (int kbi = kb0; kbi < kb1; ++kbi) {
        __syncthreads();
        for (int idx = tid; idx < kTileN * kTileK; idx += 128) {
          const int r = idx / kTileK, k = idx % kTileK;
          Ws[r * (kTileK + 1) + k] = load_w(a.W, (long)(T * kTileN + r) * a.K + kbi * kTileK + k, a.e.g.wtype);
        }
        for (int idx = tid; idx < kSimtTok * kTileK; idx += 128) {
          const int t = idx / kTileK, k = idx % kTileK;
          Xs[idx] = (tok0 + t < a.e.n_tok) ? load_x(a, a.e.tok_base + tok0 + t, kbi * kTileK + k) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kTileK; ++k) {
          const float w = Ws[tid * (kTileK + 1) + k];
#pragma unroll
          for (int t = 0; t < kSimtTok; ++t) acc[t] = fmaf(w, Xs[t * kTileK + k], acc[t]);
        }
      }
      if (a.omode == O_RED) {
        float* dcol = a.dst + (long)(a.e.tok_base + tok0) * a.dst_ld + T * kTileN + tid;
        const float wsc = a.e.wscale ? a.e.wscale[T * kTileN + tid] : 1.f;
#pragma unroll
        for (int t = 0; t < kSimtTok; ++t)
          if (tok0 + t < a.e.n_tok) atomicAdd(dcol + (long)t * a.dst_ld, acc[t] * wsc);
      } else {
        acc_add16(acc_tile + (long)tid * nt, tok0, a.e.n_tok, acc);
      }
    }
    if (a.omode == O_RED) {
      u = seg_end;
      continue;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int c_lo = p.owner(T * p.kb), c_hi = p.owner((T + 1) * p.kb - 1);
      const int old = atomicAdd(a.counters + T, 1);
      s_last = (old == c_hi - c_lo);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      tile_epilogue(a.e, T, acc_tile, nt, smem, tid);
      if (tid == 0) a.counters[T] = 0;
    }
    u = seg_end;
  }
}

void launch_gemm_simt(const GemmArgs& a, cudaStream_t s) {
  launch_pdl(gemm_simt_kernel, dim3(a.p.grid), dim3(128), 0, s, a);
}

// ------------------------------------------------------------------ attention (CUDA cores)
__device__ __forceinline__ float load_kv(const void* base, long idx, int kvtype) {
  if (kvtype == KV_F32) return reinterpret_cast<const float*>(base)[idx];
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
}

__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  pdl_wait();
  pdl_launch_dependents();
  const Geo& g = a.g;
  const int d = g.d, R = g.G * kBlock, dp = d + 1;
  float* Qs = sm;                 // [R][d+1]
  float* Os = Qs + R * dp;        // [R][d+1]
  float* Ks = Os + R * dp;        // [64][d+1]
  float* Vs = Ks + kPage * dp;    // [d][65]
  const int tid = threadIdx.x;
  const int item = blockIdx.x;
  int s, kvh, k0, k1;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1);
  const int slot = a.rd->seq_slot[s];
  for (int idx = tid; idx < R * d; idx += 128) {
    const int r = idx / d, dim = idx % d;
    const int i = r / g.G, hl = r % g.G;      // row = token * G + local head
    const long qi = ((long)(s * kBlock + i) * g.Hq + kvh * g.G + hl) * d + dim;
    Qs[r * dp + dim] = load_kv(a.q, qi, g.kvtype);
    Os[r * dp + dim] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const bool active = tid < R;
  for (int kp = k0; kp < k1; kp += kPage) {
    const int pidx = kp / kPage;
    const int page = a.block_table[(long)slot * g.pages_per_seq + pidx];
    const int kc = min(kPage, k1 - kp);
    __syncthreads();
    if (page < 0 || page >= g.max_pages) {
      if (tid == 0) atomicExch(a.err, DERR_BAD_PAGE);
      break;
    }
    for (int idx = tid; idx < kPage * d; idx += 128) {
      const int j = idx / d, dim = idx % d;
      Ks[j * dp + dim] = j < kc ? load_kv(a.kpool, k_index(g, a.layer, page, kvh, j, dim), g.kvtype) : 0.f;
      const int dv = idx / kPage, jv = idx % kPage;
      Vs[dv * (kPage + 1) + jv] = jv < kc ? load_kv(a.vpool, v_index(g, a.layer, page, kvh, jv, dv), g.kvtype) : 0.f;
    }
    __syncthreads();
    if (active) {
      float sc[kPage];
      float mx = m;
#pragma unroll
      for (int j = 0; j < kPage; ++j) {
        float acc = 0.f;
        if (j < kc) {
          for (int dim = 0; dim < d; ++dim) acc = fmaf(Qs[tid * dp + dim], Ks[j * dp + dim], acc);
          acc *= a.scale_log2;
          mx = fmaxf(mx, acc);
        }
        sc[j] = acc;
      }
      const float alpha = exp2f(m - mx);
      float lsum = 0.f;
#pragma unroll
      for (int j = 0; j < kPage; ++j) {
        sc[j] = j < kc ? exp2f(sc[j] - mx) : 0.f;
        lsum += sc[j];
      }
      l = l * alpha + lsum;
      m = mx;
      for (int dim = 0; dim < d; ++dim) {
        float acc = Os[tid * dp + dim] * alpha;
#pragma unroll
        for (int j = 0; j < kPage; ++j) acc = fmaf(sc[j], Vs[dim * (kPage + 1) + j], acc);
        Os[tid * dp + dim] = acc;
      }
    }
  }
  __syncthreads();
  const long ob = (long)item * R;
  for (int idx = tid; idx < R * d; idx += 128) {
    const int r = idx / d, dim = idx % d;
    a.part_o[(ob + r) * d + dim] = Os[r * dp + dim];
  }
  if (active) {
    a.part_ml[(ob + tid) * 2 + 0] = m;
    a.part_ml[(ob + tid) * 2 + 1] = l;
  }
}

void launch_attention_simt(const AttnArgs& a, int n_items, cudaStream_t s) {
  const int R = a.g.G * kBlock, dp = a.g.d + 1;
  const size_t smem = sizeof(float) * (2 * R * dp + kPage * dp + a.g.d * (kPage + 1));
  cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(attn_simt_kernel, dim3(n_items), dim3(128), smem, s, a);
}

// Merge the split-KV partials of one (token, q head) row into the O-proj operand.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const Geo& g = a.g;
  const int row = blockIdx.x;               // tok * Hq + h
  const int tok = row / g.Hq, h = row % g.Hq;
  const int s = tok / kBlock, i = tok % kBlock;
  const int kvh = h / g.G, hl = h % g.G;
  const int R = g.G * kBlock, r = i * g.G + hl;
  const RoundDesc* rd = a.rd;
  const int nsplit = (rd->item0[s + 1] - rd->item0[s]) / g.Hkv;
  const int it0 = rd->item0[s] + kvh * nsplit;
  float M = -INFINITY;
  for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, a.part_ml[((long)(it0 + sp) * R + r) * 2]);
  const int dim = threadIdx.x;
  if (dim >= g.d) return;
  float num = 0.f, den = 0.f;
  for (int sp = 0; sp < nsplit; ++sp) {
    const long pr = (long)(it0 + sp) * R + r;
    const float w = exp2f(a.part_ml[pr * 2] - M);
    den += w * a.part_ml[pr * 2 + 1];
    num += w * a.part_o[pr * g.d + dim];
  }
  put_operand(a.op, (long)tok * a.op_ld + h * g.d + dim, a.op_plane, num / den, a.op_f32);
}

void launch_attn_combine(const AttnArgs& a, int n_tok, cudaStream_t s) {
  launch_pdl(attn_combine_kernel, dim3(n_tok * a.g.Hq), dim3(128), 0, s, a);
}

// ------------------------------------------------------------------ per-call init
// CTA r < n_rows: stage row r (residual stream + operand); CTA n_rows: upload
// the descriptor, apply page-table entries and clear accumulators.
__global__ void __launch_bounds__(128) init_kernel(InitArgs a, InitBlob b) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x, tid = threadIdx.x;
  if (r == a.n_rows) {
    const int* src = reinterpret_cast<const int*>(&b);
    int* dst = reinterpret_cast<int*>(a.desc_dst);
    for (int i = tid; i < a.desc_bytes / 4; i += blockDim.x) dst[i] = src[i];
    for (int i = tid; i < b.n_pt; i += blockDim.x) a.block_table[b.pt_idx[i]] = b.pt_page[i];
    for (int i = tid; i < a.zero_n; i += blockDim.x) a.zero_ptr[i] = 0.f;
    return;
  }
  // RoPE (cos, sin) of this row's position, mscale folded in
  const int pos = a.is_round ? b.round.pos[r] : b.ingest.row_pos[r];
  const int half = a.g.d / 2;
  for (int j = tid; j < half; j += blockDim.x) {
    float sn, cs;
    rope_sincos(pos, a.inv_freq, j, &sn, &cs);
    a.rope_cs[(long)r * half + j] = make_float2(cs * a.g.mscale, sn * a.g.mscale);
  }
  for (int c = tid; c < a.width; c += blockDim.x) {
    const float v = a.src[(long)r * a.width + c];
    if (a.h) a.h[(long)r * a.width + c] = v;
    else put_operand(a.op, (long)r * a.op_ld + c, a.op_plane, v, a.op_f32);
  }
}

void launch_init(const InitArgs& a, const InitBlob& blob, cudaStream_t s) {
  launch_pdl(init_kernel, dim3(a.n_rows + 1), dim3(128), 0, s, a, blob);
}

__global__ void __launch_bounds__(128) final_norm_kernel(const float* h, const float* gain, float* out, int H,
                                                         float eps) {
  pdl_wait();
  pdl_launch_dependents();
  const int tok = blockIdx.x, tid = threadIdx.x;
  __shared__ float red[4];
  float ss = 0.f;
  for (int c = tid; c < H; c += blockDim.x) {
    const float v = h[(long)tok * H + c];
    ss += v * v;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  const float r = rsqrtf((red[0] + red[1] + red[2] + red[3]) / (float)H + eps);
  for (int c = tid; c < H; c += blockDim.x) out[(long)tok * H + c] = h[(long)tok * H + c] * gain[c] * r;
}

void launch_final_norm(const float* h, const float* gain, float* out, int n_tok, const Geo& g, cudaStream_t s) {
  launch_pdl(final_norm_kernel, dim3(n_tok), dim3(128), 0, s, h, gain, out, g.H, g.eps);
}

__global__ void kv_read_kernel(Geo g, const void* kpool, const void* vpool, const int* block_table,
                               int slot, int layer, int row0, float* k_out, float* v_out) {
  pdl_wait();
  const int rr = blockIdx.x, row = row0 + rr;
  const int page = block_table[(long)slot * g.pages_per_seq + row / kPage];
  const int off = row % kPage;
  for (int idx = threadIdx.x; idx < g.Hkv * g.d; idx += blockDim.x) {
    const int head = idx / g.d, dim = idx % g.d;
    k_out[(long)rr * g.Hkv * g.d + idx] = load_kv(kpool, k_index(g, layer, page, head, off, dim), g.kvtype);
    v_out[(long)rr * g.Hkv * g.d + idx] = load_kv(vpool, v_index(g, layer, page, head, off, dim), g.kvtype);
  }
}

void launch_kv_read(const Geo& g, const void* kpool, const void* vpool, const int* block_table, int slot,
                    int layer, int row0, int nrows, float* k_out, float* v_out, cudaStream_t s) {
  if (nrows > 0) kv_read_kernel<<<nrows, 128, 0, s>>>(g, kpool, vpool, block_table, slot, layer, row0, k_out, v_out);
}

}  // namespace dfl
