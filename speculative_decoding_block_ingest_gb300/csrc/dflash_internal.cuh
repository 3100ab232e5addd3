// dflash_internal.cuh -- device-side structures and the shared GEMM epilogue.
//
// Every projection of the drafter is a "swap-AB" weight-streaming product:
// the weight's output features are the tile rows (128 per tile) and the
// (few) token rows are the columns.  A tile's K range is split over CTAs
// (stream-K over units of 64 K-columns).  Each contributor adds its f32
// partial into the tile's accumulator with fire-and-forget reductions
// (red.global.add), fences, and takes a ticket; the last one to arrive reads
// the accumulated tile once (and clears it for the next call) and runs the
// tile's fused epilogue (norm scale, head RMSNorm + RoPE, SwiGLU, residual,
// KV-page write).
//
// The last arriver's epilogue sits on the kernel's critical path and runs
// once per SM on cold instruction caches, so it is kept short and loop-shaped:
// per-token constants (RoPE cos/sin, KV destination rows) are prepared
// beforehand by the per-call init kernels and the host, and no global load in
// it waits on another.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dfl {

constexpr int kBlock = 16;        // block rows per sequence (gamma = 16)
constexpr int kPage = 64;         // KV rows per page
constexpr int kTileN = 128;       // weight rows per tile
constexpr int kTileK = 64;        // K columns per unit
constexpr int kPassTok = 256;     // token columns per GEMM pass (one MMA N)
constexpr int kMaxBatch = 64;
constexpr int kMaxIngestRows = 512;
constexpr int kMaxConvGroups = 256;   // DFlash2 conv channel groups
constexpr int kMaxHidden = 8192;  // widest residual row the row kernels hold in registers
constexpr int kMaxPtUpdates = 160;
constexpr int kMaxItems = 2048;   // attention work items of a round
constexpr int kEpiThreads = 128;  // threads running a tile epilogue
constexpr int kEpiTokChunk = 32;  // tokens per epilogue pass
constexpr int kEpiBar = 1;        // named barrier id used by the epilogue
// Two e4m3 codes, in bytes 0 and 2 of t (bytes 1 and 3 zero), as two f16
// values scaled by 2^-8 (low half first).  For a code b = s eeee mmm the f16
// pattern s 0 eeee mmm 0000000 (b << 7 with the sign moved up one bit, i.e.
// (b + (b & 0x80)) << 7) has exponent field e against f16's bias 15 instead
// of e4m3's 7 and the same mantissa, so it is the value times 2^-8 for the
// normal codes, and for the subnormal ones (e = 0) both formats scale the
// mantissa alike.  Exact for every finite code (neither the weights nor the
// cache ever hold a NaN code).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t t) {
  return (t + (t & 0x00800080u)) << 7;
}

// Codes (b0 b1 b2 b3) of a word as the f16 pairs (b0, b1) and (b2, b3),
// scaled by 2^-8 (integer operations only).
__device__ __forceinline__ uint2 e4m3x4_to_f16x4_scaled(uint32_t w) {
  return make_uint2(e4m3x2_to_f16x2_scaled(__byte_perm(w, 0u, 0x4140)), e4m3x2_to_f16x2_scaled(__byte_perm(w, 0u, 0x4342)));
}

// e4m3 weights and cached K/V reach the tensor cores as f16 values scaled by
// 2^-8 (the kernels widen the codes with integer operations); the row
// scales, multiplied by this, undo it exactly.
constexpr float kW8Unscale = 256.f;
constexpr int kRedFloats = kEpiTokChunk * (kTileN + 1) + kEpiTokChunk;   // epilogue shared scratch

enum WType { W_F32 = 0, W_BF16 = 1, W_FP8 = 2 };
// KV cache element: f32, bf16, or OCP e4m3 codes with one f32 scale per
// (layer, page row, kv head) for K and for V.
enum KvType { KV_F32 = 0, KV_BF16 = 1, KV_FP8 = 2 };
// Fused tile epilogues of the ingest's projections.
enum EpiKind { EPI_FC = 0, EPI_KV = 1 };
enum DevErr { DERR_NONE = 0, DERR_TIMEOUT = 4, DERR_BAD_PAGE = 6 };

// Optional launch trace.  Per CTA, kTraceWords u64: {smid, %globaltimer at
// entry (ns), SM clock64 cycles since entry at fixed points 1..13 of the
// kernel (see each kernel), %globaltimer at exit}.  Points written by one
// warp compare exactly; points of different warps only roughly.
constexpr int kTraceWords = 16;
__device__ __forceinline__ unsigned long long trace_clock() {
  unsigned long long c;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(c)::"memory");
  return c;
}
__device__ __forceinline__ void trace_entry(unsigned long long* tr, int cta, unsigned long long* c0) {
  *c0 = trace_clock();
  if (tr) {
    unsigned int smid;
    unsigned long long t;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    tr[(long)cta * kTraceWords] = smid;
    tr[(long)cta * kTraceWords + 1] = t;
    tr[(long)cta * kTraceWords + kTraceWords - 1] = 0;   // exit: the warps' maximum (trace_exit_warp)
  }
}
__device__ __forceinline__ void trace_mark(unsigned long long* tr, int cta, int point, unsigned long long c0) {
  if (tr) {
    const unsigned long long v = trace_clock() - c0;
    asm volatile("st.global.u64 [%0], %1;" ::"l"(tr + (long)cta * kTraceWords + 1 + point), "l"(v) : "memory");
  }
}
// A measured quantity (e.g. cycles spent waiting) at point `point`.
__device__ __forceinline__ void trace_put(unsigned long long* tr, int cta, int point, unsigned long long v) {
  if (tr) asm volatile("st.global.u64 [%0], %1;" ::"l"(tr + (long)cta * kTraceWords + 1 + point), "l"(v) : "memory");
}
// %globaltimer (ns) at the CTA's exit in the last word (after point 13).
__device__ __forceinline__ void trace_exit(unsigned long long* tr, int cta) {
  if (tr) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    asm volatile("st.global.u64 [%0], %1;" ::"l"(tr + (long)cta * kTraceWords + kTraceWords - 1), "l"(t) : "memory");
  }
}
// Entry and exit stamps of the element-wise kernels (thread 0 of each CTA).
// The CTA's exit as the latest of its warps' finishing times: lane 0 of every
// warp takes the maximum into the exit word (zeroed by trace_entry before the
// CTA's set-up barrier).  A single
// thread's stamp after the final barrier can read early: the role warps of
// the pipelined kernels reach that barrier converged only in appearance, so
// the first thread past it is no proof that the others are done.
__device__ __forceinline__ void trace_exit_warp(unsigned long long* tr, int cta) {
  if (tr && (threadIdx.x & 31) == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    atomicMax(tr + (long)cta * kTraceWords + kTraceWords - 1, t);
  }
}
__device__ __forceinline__ void trace_cta_entry(unsigned long long* tr) {
  unsigned long long c0;
  if (tr && threadIdx.x == 0) trace_entry(tr, blockIdx.x, &c0);
}
__device__ __forceinline__ void trace_cta_exit(unsigned long long* tr) {
  if (tr && threadIdx.x == 0) trace_exit(tr, blockIdx.x);
}

// Per-call descriptor of a drafting round (device copy lives in the workspace).
struct RoundDesc {
  int n_seq, n_tok, split_pages, n_items;
  int seq_slot[kMaxBatch];
  int len[kMaxBatch];
  int item0[kMaxBatch + 1];        // attention work items of seq s: [item0[s], item0[s+1])
  int kstart[kMaxBatch];           // first attended key position (context window; 0 = all)
  int pos[kMaxBatch * kBlock];     // absolute position of each block row
  int dest[kMaxBatch * kBlock];    // page*64 + offset of the row's transient K/V
  uint16_t perm[kMaxItems];        // launch order: attention CTA c runs work item perm[c]
};

// Per-call descriptor of an ingest (rows in call order).
struct IngestDesc {
  int n_rows;
  int row_pos[kMaxIngestRows];     // absolute position
  int row_dest[kMaxIngestRows];    // page*64 + offset of the row's cached K/V
};

// Kernel-parameter blob of an init kernel: the descriptor plus page-table
// entries to apply (flat index into the block table -> page id).
struct InitBlob {
  union {
    RoundDesc round;
    IngestDesc ingest;
  };
  int n_pt;
  int pt_idx[kMaxPtUpdates];
  int pt_page[kMaxPtUpdates];
};

// Constant model geometry shared by kernels.
struct Geo {
  int L, H, Hq, Hkv, d, I, n, G;
  int qkv_n, kv_n;      // (Hq+2Hkv)*d ; 2*Hkv*d
  int Mt;               // token-row capacity of activation buffers
  int wtype, kvtype;
  int max_pages, pages_per_seq;
  float eps, mscale;
};

// Epilogue arguments of one GEMM call site.
struct EpiArgs {
  int kind;                   // EpiKind
  int n_tok;                  // token columns of this pass
  int tok_base;               // first token of this pass
  const float* wscale;        // per weight row scale of e4m3 weights (times kW8Unscale), or null
  const float* ss_in;         // KV: per token sum of squares -> rsqrt(ss/H+eps) scale; null = 1
  float* ss_out;              // FC: per token sum of squares of the features
  const float* gain;          // FC: hidden_norm gain
  void* op;                   // FC: operand written for the K/V projection (hi/lo bf16 planes or f32)
  int op_ld;
  long op_plane;              // elements between hi and lo planes
  int op_kind;                 // operand kind (OpKind)
  const float* kn;            // KV: k head-norm gains [L][d]
  void* kpool;                // K pool base (all layers)
  void* vpool;                // V^T pool base (all layers)
  const int* dest;            // KV: per token page*64+offset (descriptor copy)
  const float2* rope_cs;      // KV: per token [d/2] (cos, sin), mscale folded in
  int* err;
  Geo g;
};

// Stream-K partition of one GEMM: CTA c owns units [start(c), start(c+1)).
struct Part {
  int units, grid, kb;        // total units, CTAs, units per tile
  __host__ __device__ int start(int c) const { return (int)(((long long)c * units) / grid); }
  // the CTA that owns unit u
  __host__ __device__ int owner(int u) const { return (int)((((long long)u + 1) * grid - 1) / units); }
};

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Named barrier of the epilogue threads.  The non-aligned form counts each
// arriving thread, so it stays correct when lanes reach it at different times
// (after per-lane work such as the stream-K ticket).
__device__ __forceinline__ void epi_sync() {
  asm volatile("barrier.sync %0, %1;" ::"r"(kEpiBar), "r"(kEpiThreads) : "memory");
}

// Operand element types of the projections: hi/lo bf16 planes beside bf16
// weights, f32 for the f32 drafter, hi/lo f16 planes beside e4m3 weights
// (widened to f16 for the tensor cores, which take one type for both sides).
enum OpKind { OPK_BF16 = 0, OPK_F32 = 1, OPK_F16 = 2 };

__device__ __forceinline__ void put_operand(void* op, long idx, long plane, float v, int kind) {
  if (kind == OPK_F32) {
    reinterpret_cast<float*>(op)[idx] = v;
  } else if (kind == OPK_F16) {
    const __half hi = __float2half_rn(v);
    const __half lo = __float2half_rn(v - __half2float(hi));
    reinterpret_cast<__half*>(op)[idx] = hi;
    reinterpret_cast<__half*>(op)[idx + plane] = lo;
  } else {
    __nv_bfloat16 hi = __float2bfloat16_rn(v);
    __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    reinterpret_cast<__nv_bfloat16*>(op)[idx] = hi;
    reinterpret_cast<__nv_bfloat16*>(op)[idx + plane] = lo;
  }
}

// Four consecutive operand elements [idx, idx + 4) as one vector store per
// plane (idx and plane multiples of 4); the values put_operand would store.
__device__ __forceinline__ void put_operand4(void* op, long idx, long plane, float4 v, int kind) {
  if (kind == OPK_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(op) + idx) = v;
    return;
  }
  const float x[4] = {v.x, v.y, v.z, v.w};
  uint32_t hi[2], lo[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (kind == OPK_F16) {
      const __half h0 = __float2half_rn(x[2 * p]), h1 = __float2half_rn(x[2 * p + 1]);
      const __half l0 = __float2half_rn(x[2 * p] - __half2float(h0));
      const __half l1 = __float2half_rn(x[2 * p + 1] - __half2float(h1));
      hi[p] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      lo[p] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    } else {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(x[2 * p]), h1 = __float2bfloat16_rn(x[2 * p + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(x[2 * p] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(x[2 * p + 1] - __bfloat162float(h1));
      hi[p] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[p] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
  }
  uint16_t* base = reinterpret_cast<uint16_t*>(op);
  *reinterpret_cast<uint2*>(base + idx) = make_uint2(hi[0], hi[1]);
  *reinterpret_cast<uint2*>(base + idx + plane) = make_uint2(lo[0], lo[1]);
}

__device__ __forceinline__ void put_kv(void* base, long idx, float v, int kvtype) {
  if (kvtype == KV_F32) reinterpret_cast<float*>(base)[idx] = v;
  else reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

// PER consecutive elements of a bf16 or f32 row [idx, idx + PER) (idx a
// multiple of PER): one vector store at PER = 4, else element by element.
template <int PER>
__device__ __forceinline__ void put_kv_row(void* base, long idx, const float* x, int kvtype) {
  if (PER == 4 && kvtype == KV_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = make_float4(x[0], x[1], x[2], x[3]);
  } else if (PER == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(base) + idx) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
#pragma unroll
    for (int q = 0; q < PER; ++q) put_kv(base, idx + q, x[q], kvtype);
  }
}

__device__ __forceinline__ long pool_layer_elems(const Geo& g) {
  return (long)g.max_pages * g.Hkv * kPage * g.d;
}

// FP8 cache: each pool holds its e4m3 codes ([L][page][Hkv][64][d] for K,
// [L][page][Hkv][d][64] for V^T, one byte each) followed by its scales
// [L][page][Hkv][64] f32.
__host__ __device__ __forceinline__ long fp8_pool_codes(const Geo& g) {
  return (long)g.L * g.max_pages * g.Hkv * kPage * g.d;
}
__host__ __device__ __forceinline__ long kv_scale_index(const Geo& g, int layer, int page, int head, int off) {
  return (((long)layer * g.max_pages + page) * g.Hkv + head) * kPage + off;
}
__host__ __device__ __forceinline__ float* fp8_pool_scales(const Geo& g, void* pool) {
  return reinterpret_cast<float*>(static_cast<char*>(pool) + fp8_pool_codes(g));
}
__host__ __device__ __forceinline__ const float* fp8_pool_scales(const Geo& g, const void* pool) {
  return reinterpret_cast<const float*>(static_cast<const char*>(pool) + fp8_pool_codes(g));
}

// e4m3 scale of one head row from its absolute maximum: the largest value
// maps to the largest finite code (448); an all-zero row takes scale 1.
__device__ __forceinline__ float fp8_row_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f; }

// Two values divided by the row scale (IEEE division) and rounded to
// nearest-even e4m3 with saturation; a in the low byte.
__device__ __forceinline__ uint16_t fp8_pair(float a, float b, float s) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)), __NV_SATFINITE, __NV_E4M3);
}

// K pool: [L][page][Hkv][64][d]
__device__ __forceinline__ long k_index(const Geo& g, int layer, int page, int head, int off, int dim) {
  return layer * pool_layer_elems(g) + (((long)page * g.Hkv + head) * kPage + off) * g.d + dim;
}
// V^T pool: [L][page][Hkv][d][64]
__device__ __forceinline__ long v_index(const Geo& g, int layer, int page, int head, int off, int dim) {
  return layer * pool_layer_elems(g) + (((long)page * g.Hkv + head) * g.d + dim) * kPage + off;
}

// Store one K (kind 1) or V (kind 2) head row of the cache in e4m3 with its
// scale (PER dims per lane of a warp, lane l holds dims l*PER ..).
template <int PER>
__device__ __forceinline__ void put_row_fp8(const Geo& g, const float* x, int lane, int kind, int layer, int tok,
                                            int head, int dst, void* kpool, void* vpool) {
  (void)tok;
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) am = fmaxf(am, fabsf(x[i]));
  const float sc = fp8_row_scale(warp_max(am));
  uint8_t c[PER];
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    const uint16_t w = fp8_pair(x[i], x[i + 1], sc);
    c[i] = (uint8_t)(w & 0xFF);
    c[i + 1] = (uint8_t)(w >> 8);
  }
  const int dim0 = lane * PER;
  const int page = dst >> 6, off = dst & (kPage - 1);
  if (kind == 1) {
    uint8_t* row = static_cast<uint8_t*>(kpool) + k_index(g, layer, page, head, off, dim0);
#pragma unroll
    for (int i = 0; i < PER; ++i) row[i] = c[i];
    if (lane == 0) fp8_pool_scales(g, kpool)[kv_scale_index(g, layer, page, head, off)] = sc;
  } else {
    uint8_t* vp = static_cast<uint8_t*>(vpool);
#pragma unroll
    for (int i = 0; i < PER; ++i) vp[v_index(g, layer, page, head, off, dim0 + i)] = c[i];
    if (lane == 0) fp8_pool_scales(g, vpool)[kv_scale_index(g, layer, page, head, off)] = sc;
  }
}

// NeoX rotation angle for pair j at position p, reduced to [-pi, pi] in f64
// (positions reach ~66k, where an f32 product would be off by ~1e-2 rad).
__device__ __forceinline__ void rope_sincos(int pos, const double* inv_freq, int j, float* s, float* c) {
  double th = (double)pos * inv_freq[j];
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  th = fma(-two_pi, rint(th * inv_two_pi), th);
  sincosf((float)th, s, c);
}

// Locate attention work item `item`: sequence s, kv head, and its key range
// [k0, k1) within [cached context ; 16 block rows], splits counted from the
// page holding the sequence's first attended key ks (keys below ks, in that
// first page only, are masked by the kernels).
__device__ __forceinline__ void attn_item(const RoundDesc* rd, int Hkv, int item, int* s_out, int* g_out,
                                          int* k0, int* k1, int* ks = nullptr) {
  int s = 0;
  while (s + 1 < rd->n_seq && rd->item0[s + 1] <= item) ++s;
  const int local = item - rd->item0[s];
  const int nsplit = (rd->item0[s + 1] - rd->item0[s]) / Hkv;
  const int g = local / nsplit, sp = local % nsplit;
  const int n_keys = rd->len[s] + kBlock;
  const int base = rd->kstart[s] / kPage * kPage;
  *s_out = s;
  *g_out = g;
  *k0 = base + sp * rd->split_pages * kPage;
  *k1 = min(n_keys, base + (sp + 1) * rd->split_pages * kPage);
  if (ks) *ks = rd->kstart[s];
}

// ------------------------------------------------------------------ stream-K reduction
// Tile accumulator layout: acc[tile][128 features][nt tokens] f32 (nt = the
// pass's tokens rounded up to 16), so a thread owning feature f adds and
// reads its tokens as contiguous float4s.

// Add one contributor's values v[0..15] (tokens j0..j0+15 of one feature).
__device__ __forceinline__ void acc_add16(float* acc_f, int j0, int n_tok, const float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (j0 + 4 * q < n_tok) {
      float* p = acc_f + j0 + 4 * q;
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v[4 * q]), "f"(v[4 * q + 1]),
                   "f"(v[4 * q + 2]), "f"(v[4 * q + 3])
                   : "memory");
    }
  }
}

// ------------------------------------------------------------------ epilogue
// Head-wise epilogue (K/V of an ingest, every layer) on a reduced chunk
// red[t][0..127] for tokens tok0 .. tok0+tc-1.  One warp per (token, head);
// lane l holds PER = d/32 consecutive dims, lanes 0..15 the first half (so a
// dim's RoPE partner j + d/2 sits in lane l + 16).  Every global load of a
// task is issued before any of its stores.
template <int PER>
static __device__ void epi_heads_t(const EpiArgs& e, int tile, const float* red, const float* rsc, int tok0, int tc,
                                   int et) {
  const Geo& g = e.g;
  constexpr int d = 32 * PER, half = d / 2, heads_in_tile = kTileN / d;
  const int warp = et >> 5, lane = et & 31;
  const int dim0 = lane * PER;
  const int tasks = tc * heads_in_tile;
  for (int task = warp; task < tasks; task += kEpiThreads / 32) {
    const int t = task / heads_in_tile, sh = task % heads_in_tile;
    const int tok = e.tok_base + tok0 + t;     // global token index
    const int hh = (tile * kTileN) / d + sh;   // head index within the tile's GEMM rows
    // the all-layer K/V matrix stacks [k heads; v heads] per layer
    const int layer = hh / (2 * g.Hkv);
    const int j = hh % (2 * g.Hkv);
    const int kind = j < g.Hkv ? 1 : 2;        // 1 k, 2 v
    const int head = j < g.Hkv ? j : j - g.Hkv;
    // loads first: gains, (cos, sin), destination row
    float gn[PER];
    float2 cs[PER];
    const float* __restrict__ gsrc = e.kn + (long)layer * d;
    const float2* __restrict__ csrc = e.rope_cs + (long)tok * half;
    if (kind != 2) {
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        gn[q] = gsrc[dim0 + q];
        cs[q] = csrc[(dim0 + q) % half];
      }
    }
    const int dst = e.dest[tok];
    const float rs = rsc[t];
    float x[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) x[q] = red[t * (kTileN + 1) + sh * d + dim0 + q] * rs;
    if (kind != 2) {
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < PER; ++q) ss += x[q] * x[q];
      ss = warp_sum(ss);
      const float r = rsqrtf(ss / (float)d + g.eps);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const float y = x[q] * r * gn[q];
        const float partner = __shfl_xor_sync(0xffffffffu, y, 16);   // dims j <-> j + d/2
        x[q] = lane < 16 ? (y * cs[q].x - partner * cs[q].y) : (y * cs[q].x + partner * cs[q].y);
      }
    }
    if (g.kvtype == KV_FP8) {
      put_row_fp8<PER>(g, x, lane, kind, layer, tok, head, dst, e.kpool, e.vpool);
    } else {
      const int page = dst >> 6, off = dst & (kPage - 1);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        if (kind == 1) put_kv(e.kpool, k_index(g, layer, page, head, off, dim0 + q), x[q], g.kvtype);
        else put_kv(e.vpool, v_index(g, layer, page, head, off, dim0 + q), x[q], g.kvtype);
      }
    }
  }
}

static __device__ __forceinline__ void epi_heads(const EpiArgs& e, int tile, const float* red, const float* rsc,
                                                 int tok0, int tc, int et) {
  if (e.g.d == 128) epi_heads_t<4>(e, tile, red, rsc, tok0, tc, et);
  else epi_heads_t<2>(e, tile, red, rsc, tok0, tc, et);
}

// Run the fused epilogue of `tile` from its accumulator (and clear it).
// Called by all kEpiThreads threads (et = 0..127) of the CTA that arrived
// last.  acc: the tile's accumulator [128][nt]; red: kRedFloats shared floats.
static __device__ void tile_epilogue(const EpiArgs& e, int tile, float* acc, int nt, float* red, int et,
                                     unsigned long long* tr = nullptr, int cta = 0, unsigned long long c0 = 0) {
  const Geo& g = e.g;
  float* rsc = red + kEpiTokChunk * (kTileN + 1);   // per-token input-norm scale
  const int f = et;                                 // feature within the tile
  const float wsc = e.wscale ? kW8Unscale * e.wscale[tile * kTileN + f] : 1.f;
  float* acc_f = acc + (long)f * nt;
  for (int tok0 = 0; tok0 < e.n_tok; tok0 += kEpiTokChunk) {
    const int tc = min(kEpiTokChunk, e.n_tok - tok0);
    // one batch of independent vector loads, then clear the accumulator
    float4 v[kEpiTokChunk / 4];
#pragma unroll
    for (int q = 0; q < kEpiTokChunk / 4; ++q)
      if (4 * q < tc) v[q] = __ldcg(reinterpret_cast<const float4*>(acc_f + tok0) + q);
    if (et < tc) rsc[et] = e.ss_in ? rsqrtf(e.ss_in[e.tok_base + tok0 + et] / (float)g.H + g.eps) : 1.f;
#pragma unroll
    for (int q = 0; q < kEpiTokChunk / 4; ++q) {
      if (4 * q < tc) {
        __stcg(reinterpret_cast<float4*>(acc_f + tok0) + q, make_float4(0.f, 0.f, 0.f, 0.f));
        red[(4 * q + 0) * (kTileN + 1) + f] = v[q].x * wsc;
        red[(4 * q + 1) * (kTileN + 1) + f] = v[q].y * wsc;
        red[(4 * q + 2) * (kTileN + 1) + f] = v[q].z * wsc;
        red[(4 * q + 3) * (kTileN + 1) + f] = v[q].w * wsc;
      }
    }
    if (et == 0) trace_mark(tr, cta, 11, c0);   // 11: accumulator read
    epi_sync();
    if (et == 0) trace_mark(tr, cta, 12, c0);   // 12: row scales ready
    if (e.kind == EPI_KV) {
      epi_heads(e, tile, red, rsc, tok0, tc, et);
    } else {  // EPI_FC: features c (operand c * hidden_norm gain) and their sums of squares
      const int col = tile * kTileN + f;
      const float gn = e.gain ? e.gain[col] : 1.f;
      for (int t = 0; t < tc; ++t) {
        const int tok = e.tok_base + tok0 + t;
        const float x = red[t * (kTileN + 1) + f];
        if (e.op) put_operand(e.op, (long)tok * e.op_ld + col, e.op_plane, x * gn, e.op_kind);
      }
      epi_sync();
      if (e.ss_out) {
        const int warp = et >> 5, lane = et & 31;
        for (int t = warp; t < tc; t += kEpiThreads / 32) {
          float s = 0.f;
          for (int q = 0; q < 4; ++q) {
            const float x = red[t * (kTileN + 1) + lane + 32 * q];
            s += x * x;
          }
          s = warp_sum(s);
          if (lane == 0) atomicAdd(e.ss_out + e.tok_base + tok0 + t, s);
        }
      }
    }
    if (et == 0) trace_mark(tr, cta, 13, c0);   // 13: fused step done
    epi_sync();
  }
}

}  // namespace dfl
