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
  const int item = a.rd->perm[blockIdx.x];
  int s, kvh, k0, k1, ks;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1, &ks);
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
        if (j < kc && kp + j >= ks) {
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
        sc[j] = (j < kc && kp + j >= ks) ? exp2f(sc[j] - mx) : 0.f;
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

// Merge the split-KV partials of (token, q head) rows into the O-proj
// operand.  Each row gets comb_wpr warps (1, 2, 4 or 8: enough for its
// splits) and a CTA of eight warps takes 8 / comb_wpr rows.  One pass: warp w
// of a row takes splits w, w + comb_wpr, ..., kCombDepth deep per thread,
// every (m, l) pair and partial-row load of a pass issued before the first
// use (d/4 lanes per split row); each thread merges its splits online
// against its own running maximum, and one exchange through shared memory
// merges the row's warps -- a single L2 round trip per pass.  Five deep
// covers 40 splits with eight warps (33 at one sequence of 8192): 1% faster
// there than eight deep, whose unused loads held registers.
constexpr int kCombThreads = 256;
constexpr int kCombWarps = kCombThreads / 32;
constexpr int kCombDepth = 5;

__global__ void __launch_bounds__(kCombThreads) attn_combine_kernel(AttnArgs a, int n_rows) {
  trace_cta_entry(a.trace);
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float4 wacc[kCombWarps][32];
  __shared__ float wm[kCombWarps], wl[kCombWarps];
  const Geo& g = a.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wpr = a.comb_wpr, rpc = kCombWarps / wpr;
  const int row = blockIdx.x * rpc + warp / wpr, wr = warp % wpr;   // tok * Hq + h; warp of the row
  const int lpp = g.d / 4;                  // float4 lanes of a row (16 or 32)
  float m_t = -INFINITY, den = 0.f;         // this thread's running max and weighted sum of l
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int tok = 0, h = 0;
  if (row < n_rows) {
    tok = row / g.Hq;
    h = row % g.Hq;
    const int s = tok / kBlock, i = tok % kBlock;
    const int kvh = h / g.G, hl = h % g.G;
    const int R = g.G * kBlock, r = i * g.G + hl;
    const RoundDesc* rd = a.rd;
    const int nsplit = (rd->item0[s + 1] - rd->item0[s]) / g.Hkv;
    const int it0 = rd->item0[s] + kvh * nsplit;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
    const float4* po = reinterpret_cast<const float4*>(a.part_o);
    const int spw = 32 / lpp;               // split rows a warp covers at once (1 or 2)
    const int sub = lane / lpp, d4 = lane % lpp;
    const int stride = wpr * spw;           // splits per depth step
    for (int base = wr * spw + sub; base < nsplit; base += kCombDepth * stride) {
      float4 o[kCombDepth];
      float2 m[kCombDepth];
#pragma unroll
      for (int k = 0; k < kCombDepth; ++k) {
        const int sp = base + k * stride;
        const long pr = (long)(it0 + sp) * R + r;
        o[k] = sp < nsplit ? __ldcg(po + pr * lpp + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
        m[k] = sp < nsplit ? __ldcg(ml + pr) : make_float2(-INFINITY, 0.f);
      }
      float mx = m_t;
#pragma unroll
      for (int k = 0; k < kCombDepth; ++k) mx = fmaxf(mx, m[k].x);
      if (mx == -INFINITY) continue;
      const float sc = exp2f(m_t - mx);     // 0 while m_t is still -inf
      acc.x *= sc;
      acc.y *= sc;
      acc.z *= sc;
      acc.w *= sc;
      den *= sc;
#pragma unroll
      for (int k = 0; k < kCombDepth; ++k) {
        const float w = exp2f(m[k].x - mx);   // 0 for a missing split
        acc.x += w * o[k].x;
        acc.y += w * o[k].y;
        acc.z += w * o[k].z;
        acc.w += w * o[k].w;
        den += w * m[k].y;
      }
      m_t = mx;
    }
  }
  // merge the sub-rows of a warp (d = 64: lanes l and l + 16), then the row's warps
  if (lpp == 16) {
    const float mo = __shfl_xor_sync(0xffffffffu, m_t, 16);
    const float mx = fmaxf(m_t, mo);
    const float sa = mx == -INFINITY ? 0.f : exp2f(m_t - mx), sb = mx == -INFINITY ? 0.f : exp2f(mo - mx);
    float4 ob;
    ob.x = __shfl_xor_sync(0xffffffffu, acc.x, 16);
    ob.y = __shfl_xor_sync(0xffffffffu, acc.y, 16);
    ob.z = __shfl_xor_sync(0xffffffffu, acc.z, 16);
    ob.w = __shfl_xor_sync(0xffffffffu, acc.w, 16);
    const float db = __shfl_xor_sync(0xffffffffu, den, 16);
    acc = make_float4(sa * acc.x + sb * ob.x, sa * acc.y + sb * ob.y, sa * acc.z + sb * ob.z, sa * acc.w + sb * ob.w);
    den = sa * den + sb * db;
    m_t = mx;
  }
  if (lane < lpp) wacc[warp][lane] = acc;
  if (lane == 0) {
    wm[warp] = m_t;
    wl[warp] = den;
  }
  __syncthreads();
  if (row < n_rows && wr == 0 && lane < lpp) {
    float M = -INFINITY;
    for (int w = warp; w < warp + wpr; ++w) M = fmaxf(M, wm[w]);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    for (int w = warp; w < warp + wpr; ++w) {
      const float sc = wm[w] == -INFINITY ? 0.f : exp2f(wm[w] - M);
      const float4 u = wacc[w][lane];
      t.x += sc * u.x;
      t.y += sc * u.y;
      t.z += sc * u.z;
      t.w += sc * u.w;
      l += sc * wl[w];
    }
    const float inv = 1.f / l;
    const long idx = (long)tok * a.op_ld + h * g.d + 4 * lane;
    put_operand4(a.op, idx, a.op_plane, make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv), a.op_kind);
  }
  trace_cta_exit(a.trace);
}

// Wide rounds (more than 64 rows, d = 128, at most 8 splits a row): a warp
// merges RPW consecutive rows -- one token, RPW q heads -- with the loads of
// a pass (DEPTH splits of each row) issued before the first use, so a round
// of 512 rows takes 1024 CTAs instead of 2048 with one row per warp (which
// entered the SMs over 15 µs after the attention).  Two rows of four splits
// a pass: 2.5% faster than four rows of two at 32 sequences.
template <int RPW, int DEPTH>
__global__ void __launch_bounds__(kCombThreads) attn_combine_rows_kernel(AttnArgs a, int n_rows) {
  trace_cta_entry(a.trace);
  pdl_launch_dependents();
  pdl_wait();
  const Geo& g = a.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row0 = (blockIdx.x * kCombWarps + warp) * RPW;
  if (row0 < n_rows) {
    const int tok = row0 / g.Hq, h0 = row0 % g.Hq;
    const int s = tok / kBlock, i = tok % kBlock;
    const RoundDesc* rd = a.rd;
    const int nsplit = (rd->item0[s + 1] - rd->item0[s]) / g.Hkv;
    const int R = g.G * kBlock;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
    const float4* po = reinterpret_cast<const float4*>(a.part_o);
    long pr0[RPW];   // partial row of split 0 for each of the warp's rows
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const int h = h0 + k, kvh = h / g.G, hl = h % g.G;
      pr0[k] = (long)(rd->item0[s] + kvh * nsplit) * R + i * g.G + hl;
    }
    float m_t[RPW], den[RPW];
    float4 acc[RPW];
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      m_t[k] = -INFINITY;
      den[k] = 0.f;
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int base = 0; base < nsplit; base += DEPTH) {
      float4 o[DEPTH][RPW];
      float2 m[DEPTH][RPW];
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        const bool v = base + j < nsplit;
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
          const long pr = pr0[k] + (long)(base + j) * R;
          o[j][k] = v ? __ldcg(po + pr * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
          m[j][k] = v ? __ldcg(ml + pr) : make_float2(-INFINITY, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        float mx = m_t[k];
#pragma unroll
        for (int j = 0; j < DEPTH; ++j) mx = fmaxf(mx, m[j][k].x);
        if (mx == -INFINITY) continue;
        const float sc = exp2f(m_t[k] - mx);   // 0 while m_t is still -inf
        acc[k] = make_float4(acc[k].x * sc, acc[k].y * sc, acc[k].z * sc, acc[k].w * sc);
        den[k] *= sc;
#pragma unroll
        for (int j = 0; j < DEPTH; ++j) {
          const float w = exp2f(m[j][k].x - mx);   // 0 for a missing split
          acc[k].x += w * o[j][k].x;
          acc[k].y += w * o[j][k].y;
          acc[k].z += w * o[j][k].z;
          acc[k].w += w * o[j][k].w;
          den[k] += w * m[j][k].y;
        }
        m_t[k] = mx;
      }
    }
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const float inv = 1.f / den[k];
      put_operand4(a.op, (long)tok * a.op_ld + (h0 + k) * g.d + 4 * lane, a.op_plane,
                   make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv), a.op_kind);
    }
  }
  trace_cta_exit(a.trace);
}

constexpr int kCombRowsRpw = 2, kCombRowsDepth = 4;

// Rows per warp of the wide-round merge, or 0 for the per-row kernel.
static int combine_rows_rpw(const AttnArgs& a, int n_tok) {
  return n_tok > 64 && a.g.d == 128 && a.comb_max_split <= 8 && a.g.Hq % kCombRowsRpw == 0 ? kCombRowsRpw : 0;
}

// Warps per merged row for splits of up to max_split partials each: one warp
// covers kCombDepth splits a pass (d = 128; twice that at d = 64).
int attn_combine_wpr(int max_split) {
  int w = 1;
  while (w < kCombWarps && kCombDepth * w < max_split) w *= 2;
  return w;
}

int attn_combine_grid(const AttnArgs& a, int n_tok) {
  const int rpw = combine_rows_rpw(a, n_tok);
  const int rpc = rpw ? kCombWarps * rpw : kCombWarps / a.comb_wpr;
  return (n_tok * a.g.Hq + rpc - 1) / rpc;
}

void launch_attn_combine(const AttnArgs& a, int n_tok, cudaStream_t s) {
  const dim3 grid(attn_combine_grid(a, n_tok)), block(kCombThreads);
  if (combine_rows_rpw(a, n_tok))
    launch_pdl(attn_combine_rows_kernel<kCombRowsRpw, kCombRowsDepth>, grid, block, 0, s, a, n_tok * a.g.Hq);
  else
    launch_pdl(attn_combine_kernel, grid, block, 0, s, a, n_tok * a.g.Hq);
}

// ------------------------------------------------------------------ per-call init
// The row CTAs stage rows (residual stream or operand), a row's float4s in
// chunks of kInitChunk4 per CTA; the last CTA uploads the used words of the
// descriptor, applies page-table entries and clears accumulators.  Row
// copies issue four float4 loads per thread before storing.
constexpr int kInitThreads = 256;
constexpr int kInitChunk4 = 4 * kInitThreads;   // float4 of a row per CTA: four loads per thread
__global__ void __launch_bounds__(kInitThreads) init_kernel(InitArgs a, const __grid_constant__ InitBlob b) {
  trace_cta_entry(a.trace);
  pdl_launch_dependents();
  pdl_wait();
  // CTA b < n_rows * nch: row b / nch, its float4 chunk b % nch (one load
  // batch per thread); CTA n_rows * nch: the descriptor
  const int n4 = a.width / 4, nch = (n4 + kInitChunk4 - 1) / kInitChunk4;
  const int r = blockIdx.x / nch, ch = blockIdx.x % nch, tid = threadIdx.x;
  if (r == a.n_rows) {
    const int* src = reinterpret_cast<const int*>(&b);
    int* dst = reinterpret_cast<int*>(a.desc_dst);
    for (int q = 0; q < 4; ++q)
      for (int i = tid; i < a.cp_len[q]; i += kInitThreads) dst[a.cp_off[q] + i] = src[a.cp_off[q] + i];
    for (int i = tid; i < b.n_pt; i += kInitThreads) a.block_table[b.pt_idx[i]] = b.pt_page[i];
    for (int i = tid; i < a.zero_n; i += kInitThreads) a.zero_ptr[i] = 0.f;
    trace_cta_exit(a.trace);
    return;
  }
  // RoPE (cos, sin) of this row's position, mscale folded in
  if (ch == 0) {
    const int pos = a.is_round ? b.round.pos[r] : b.ingest.row_pos[r];
    const int half = a.g.d / 2;
    for (int j = tid; j < half; j += kInitThreads) {
      float sn, cs;
      rope_sincos(pos, a.inv_freq, j, &sn, &cs);
      a.rope_cs[(long)r * half + j] = make_float2(cs * a.g.mscale, sn * a.g.mscale);
    }
  }
  const float4* src4 = reinterpret_cast<const float4*>(a.src + (long)r * a.width);
  const int c_end = min(n4, (ch + 1) * kInitChunk4);
  for (int c0 = ch * kInitChunk4 + tid; c0 < c_end; c0 += 4 * kInitThreads) {
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = c0 + k * kInitThreads;
      v[k] = c < c_end ? __ldg(src4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = c0 + k * kInitThreads;
      if (c >= c_end) break;
      if (a.h) {
        reinterpret_cast<float4*>(a.h + (long)r * a.width)[c] = v[k];
      } else {
        const long idx = (long)r * a.op_ld + 4 * c;
        put_operand4(a.op, idx, a.op_plane, v[k], a.op_kind);
      }
    }
  }
  trace_cta_exit(a.trace);
}

const void* init_kernel_entry() { return reinterpret_cast<const void*>(init_kernel); }

int init_grid(const InitArgs& a) {
  const int n4 = a.width / 4;
  return a.n_rows * ((n4 + kInitChunk4 - 1) / kInitChunk4) + 1;
}

// Both arguments travel as kernel parameters (at most 32764 bytes together).
static_assert(sizeof(InitArgs) + sizeof(InitBlob) <= 32764, "init kernel parameters exceed the launch limit");

void launch_init(const InitArgs& a, const InitBlob& blob, cudaStream_t s) {
  launch_pdl(init_kernel, dim3(init_grid(a)), dim3(kInitThreads), 0, s, a, blob);
}

__global__ void kv_read_kernel(Geo g, const void* kpool, const void* vpool, const int* block_table,
                               int slot, int layer, int row0, float* k_out, float* v_out) {
  pdl_wait();
  const int rr = blockIdx.x, row = row0 + rr;
  const int page = block_table[(long)slot * g.pages_per_seq + row / kPage];
  const int off = row % kPage;
  for (int idx = threadIdx.x; idx < g.Hkv * g.d; idx += blockDim.x) {
    const int head = idx / g.d, dim = idx % g.d;
    if (g.kvtype == KV_FP8) {
      // code (exact in f16) times the row's scale
      const long si = kv_scale_index(g, layer, page, head, off);
      const uint8_t kc = static_cast<const uint8_t*>(kpool)[k_index(g, layer, page, head, off, dim)];
      const uint8_t vc = static_cast<const uint8_t*>(vpool)[v_index(g, layer, page, head, off, dim)];
      k_out[(long)rr * g.Hkv * g.d + idx] =
          __half2float(__half(__nv_cvt_fp8_to_halfraw(kc, __NV_E4M3))) * fp8_pool_scales(g, kpool)[si];
      v_out[(long)rr * g.Hkv * g.d + idx] =
          __half2float(__half(__nv_cvt_fp8_to_halfraw(vc, __NV_E4M3))) * fp8_pool_scales(g, vpool)[si];
      continue;
    }
    k_out[(long)rr * g.Hkv * g.d + idx] = load_kv(kpool, k_index(g, layer, page, head, off, dim), g.kvtype);
    v_out[(long)rr * g.Hkv * g.d + idx] = load_kv(vpool, v_index(g, layer, page, head, off, dim), g.kvtype);
  }
}

void launch_kv_read(const Geo& g, const void* kpool, const void* vpool, const int* block_table, int slot,
                    int layer, int row0, int nrows, float* k_out, float* v_out, cudaStream_t s) {
  if (nrows > 0) kv_read_kernel<<<nrows, 128, 0, s>>>(g, kpool, vpool, block_table, slot, layer, row0, k_out, v_out);
}

}  // namespace dfl
