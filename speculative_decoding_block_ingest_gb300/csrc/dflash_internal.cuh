// dflash_internal.cuh -- device-side structures and the shared GEMM epilogue.
//
// Every projection of the drafter is a "swap-AB" weight-streaming product:
// the weight's output features are the tile rows (128 per tile) and the
// (few) token rows are the columns.  A tile's K range is split over CTAs
// (stream-K over units of 64 K-columns); each contributor writes an f32
// partial [tokens][128] and the last one to arrive reduces the partials and
// runs the tile's fused epilogue (norm scale, head RMSNorm + RoPE, SwiGLU,
// residual, KV-page write).  Both GEMM mainloops (CUDA-core for f32 weights,
// tcgen05 for bf16/fp8 weights) share this epilogue.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace dfl {

constexpr int kBlock = 16;        // block rows per sequence (gamma = 16)
constexpr int kPage = 64;         // KV rows per page
constexpr int kTileN = 128;       // weight rows per tile
constexpr int kTileK = 64;        // K columns per unit
constexpr int kMaxBatch = 64;
constexpr int kMaxIngestRows = 512;
constexpr int kMaxPtUpdates = 160;
constexpr int kEpiThreads = 128;  // threads running a tile epilogue
constexpr int kEpiTokChunk = 32;  // tokens reduced per epilogue pass
constexpr int kEpiBar = 1;        // named barrier id used by the epilogue

enum WType { W_F32 = 0, W_BF16 = 1, W_FP8 = 2 };
enum KvType { KV_F32 = 0, KV_BF16 = 1 };
enum EpiKind { EPI_FC = 0, EPI_KV = 1, EPI_QKV = 2, EPI_RESID = 3, EPI_SWIGLU = 4 };
enum DevErr { DERR_NONE = 0, DERR_TIMEOUT = 4, DERR_BAD_PAGE = 6 };

// Per-call descriptor of a drafting round (device copy lives in the workspace).
struct RoundDesc {
  int n_seq, n_tok, split_pages, n_items;
  int seq_slot[kMaxBatch];
  int len[kMaxBatch];
  int item0[kMaxBatch + 1];        // attention work items of seq s: [item0[s], item0[s+1])
  int pos[kMaxBatch * kBlock];
};

// Per-call descriptor of an ingest (rows in call order).
struct IngestDesc {
  int n_rows;
  int row_slot[kMaxIngestRows];
  int row_dst[kMaxIngestRows];
  int row_pos[kMaxIngestRows];
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
  int kind;
  int layer;
  int n_tok;                  // token columns of this pass
  int tok_base;               // first token of this pass (passes hold <= 256 tokens)
  const float* wscale;        // per weight row scale (fp8), or null
  const float* ss_in;         // per token sum of squares -> rsqrt(ss/H+eps) scale; null = 1
  float* ss_out;              // per token sum of squares of the epilogue's output
  const float* gain;          // FC: hidden_norm; RESID: next pre-norm gain (or null)
  float* h;                   // RESID: residual stream [Mt][H] f32
  int h_ld;
  void* op;                   // operand written for the next GEMM (hi/lo bf16 planes or f32)
  int op_ld;
  long op_plane;              // elements between hi and lo planes
  int op_f32;
  const float* qn;            // QKV: q head-norm gain of this layer
  const float* kn;            // QKV: k gain of this layer; KV: base of [L][d]
  void* q_out;                // QKV: q buffer [Mt][Hq][d]
  void* kpool;                // K pool base (all layers)
  void* vpool;                // V^T pool base (all layers)
  const int* block_table;
  const RoundDesc* rd;
  const IngestDesc* id;
  const double* inv_freq;     // [d/2] RoPE inverse frequencies (f64)
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
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"r"(kEpiBar), "r"(kEpiThreads) : "memory");
}

__device__ __forceinline__ void put_operand(void* op, long idx, long plane, float v, int f32) {
  if (f32) {
    reinterpret_cast<float*>(op)[idx] = v;
  } else {
    __nv_bfloat16 hi = __float2bfloat16_rn(v);
    __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    reinterpret_cast<__nv_bfloat16*>(op)[idx] = hi;
    reinterpret_cast<__nv_bfloat16*>(op)[idx + plane] = lo;
  }
}

__device__ __forceinline__ void put_kv(void* base, long idx, float v, int kvtype) {
  if (kvtype == KV_F32) reinterpret_cast<float*>(base)[idx] = v;
  else reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ long pool_layer_elems(const Geo& g) {
  return (long)g.max_pages * g.Hkv * kPage * g.d;
}
// K pool: [L][page][Hkv][64][d]
__device__ __forceinline__ long k_index(const Geo& g, int layer, int page, int head, int off, int dim) {
  return layer * pool_layer_elems(g) + (((long)page * g.Hkv + head) * kPage + off) * g.d + dim;
}
// V^T pool: [L][page][Hkv][d][64]
__device__ __forceinline__ long v_index(const Geo& g, int layer, int page, int head, int off, int dim) {
  return layer * pool_layer_elems(g) + (((long)page * g.Hkv + head) * g.d + dim) * kPage + off;
}

// NeoX rotation angle for pair j at position p, reduced to [-pi, pi] in f64.
__device__ __forceinline__ void rope_sincos(int pos, const double* inv_freq, int j, float* s, float* c) {
  double th = (double)pos * inv_freq[j];
  const double two_pi = 6.283185307179586476925286766559;
  th -= two_pi * rint(th / two_pi);
  sincosf((float)th, s, c);
}

// ------------------------------------------------------------------ epilogue
// Head-wise epilogue (QKV of a round, K/V of an ingest) on a reduced chunk
// red[t][0..127] for tokens tok0 .. tok0+tc-1.  One warp per (token, head).
static __device__ void epi_heads(const EpiArgs& e, int tile, const float* red, int tok0, int tc, int et) {
  const Geo& g = e.g;
  const int d = g.d;
  const int per = d / 32;                 // values per lane
  const int heads_in_tile = kTileN / d;
  const int warp = et >> 5, lane = et & 31;
  const int tasks = tc * heads_in_tile;
  for (int task = warp; task < tasks; task += kEpiThreads / 32) {
    const int t = task / heads_in_tile, sh = task % heads_in_tile;
    const int tok = e.tok_base + tok0 + t;      // global token index
    const int hh = (tile * kTileN) / d + sh;   // head index within the tile's GEMM rows
    int layer, kind, head;                     // kind 0 q, 1 k, 2 v
    int pos, slot, row;
    if (e.kind == EPI_QKV) {
      layer = e.layer;
      if (hh < g.Hq) { kind = 0; head = hh; }
      else if (hh < g.Hq + g.Hkv) { kind = 1; head = hh - g.Hq; }
      else { kind = 2; head = hh - g.Hq - g.Hkv; }
      const int s = tok / kBlock;
      pos = e.rd->pos[tok];
      slot = e.rd->seq_slot[s];
      row = e.rd->len[s] + (tok % kBlock);
    } else {
      layer = hh / (2 * g.Hkv);
      const int j = hh % (2 * g.Hkv);
      kind = j < g.Hkv ? 1 : 2;
      head = j < g.Hkv ? j : j - g.Hkv;
      pos = e.id->row_pos[tok];
      slot = e.id->row_slot[tok];
      row = e.id->row_dst[tok];
    }
    float rs = 1.f;
    if (e.ss_in) rs = rsqrtf(e.ss_in[tok] / (float)g.H + g.eps);
    float x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < per) x[q] = red[t * (kTileN + 1) + sh * d + lane * per + q] * rs;
    if (kind != 2) {
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < per) ss += x[q] * x[q];
      ss = warp_sum(ss);
      const float r = rsqrtf(ss / (float)d + g.eps);
      const float* gn = (kind == 0) ? e.qn : (e.kind == EPI_QKV ? e.kn : e.kn + (long)layer * d);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < per) x[q] = x[q] * r * gn[lane * per + q];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < per) {
          const float partner = __shfl_xor_sync(0xffffffffu, x[q], 16);
          const int dim = lane * per + q;
          const int j = dim % (d / 2);
          float sn, cs;
          rope_sincos(pos, e.inv_freq, j, &sn, &cs);
          x[q] = (lane < 16 ? (x[q] * cs - partner * sn) : (x[q] * cs + partner * sn)) * g.mscale;
        } else {
          (void)__shfl_xor_sync(0xffffffffu, 0.f, 16);
        }
      }
    }
    if (kind == 0) {
      const long base = ((long)tok * g.Hq + head) * d;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < per) put_kv(e.q_out, base + lane * per + q, x[q], g.kvtype);
    } else {
      const int page = e.block_table[(long)slot * g.pages_per_seq + row / kPage];
      const int off = row % kPage;
      if (page < 0 || page >= g.max_pages) {
        if (lane == 0) atomicExch(e.err, DERR_BAD_PAGE);
        continue;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < per) {
          const int dim = lane * per + q;
          if (kind == 1) put_kv(e.kpool, k_index(g, layer, page, head, off, dim), x[q], g.kvtype);
          else put_kv(e.vpool, v_index(g, layer, page, head, off, dim), x[q], g.kvtype);
        }
      }
    }
  }
}

// Reduce the partials of `tile` (contributors c_lo..c_hi, slot c+tile) and
// run its epilogue.  Called by all kEpiThreads threads (et = 0..127) of the
// CTA that arrived last.  red: shared scratch [kEpiTokChunk][129] floats.
static __device__ void tile_epilogue(const EpiArgs& e, int tile, int c_lo, int c_hi, const float* part,
                              float* red, int et) {
  const Geo& g = e.g;
  const long slot_elems = (long)g.Mt * kTileN;
  const int f = et;                                 // feature within the tile
  const int row = tile * kTileN + f;                // weight row
  const float wsc = e.wscale ? e.wscale[row] : 1.f;
  for (int tok0 = 0; tok0 < e.n_tok; tok0 += kEpiTokChunk) {
    const int tc = min(kEpiTokChunk, e.n_tok - tok0);
    for (int t = 0; t < tc; ++t) {
      float v = 0.f;
      for (int c = c_lo; c <= c_hi; ++c)
        v += __ldcg(part + (long)(c + tile) * slot_elems + (long)(tok0 + t) * kTileN + f);
      red[t * (kTileN + 1) + f] = v * wsc;
    }
    epi_sync();
    if (e.kind == EPI_QKV || e.kind == EPI_KV) {
      epi_heads(e, tile, red, tok0, tc, et);
    } else if (e.kind == EPI_SWIGLU) {
      // tile rows [0,64) = gate rows, [64,128) = up rows of act columns [64*tile, 64*tile+64)
      const int j = et & 63;
      for (int t = et >> 6; t < tc; t += 2) {
        const int tok = e.tok_base + tok0 + t;
        const float rs = e.ss_in ? rsqrtf(e.ss_in[tok] / (float)g.H + g.eps) : 1.f;
        const float gv = red[t * (kTileN + 1) + j] * rs;
        const float uv = red[t * (kTileN + 1) + 64 + j] * rs;
        const float a = gv / (1.f + expf(-gv)) * uv;
        put_operand(e.op, (long)tok * e.op_ld + tile * 64 + j, e.op_plane, a, e.op_f32);
      }
    } else {  // EPI_FC, EPI_RESID
      const int col = tile * kTileN + f;
      for (int t = 0; t < tc; ++t) {
        const int tok = e.tok_base + tok0 + t;
        float v = red[t * (kTileN + 1) + f];
        if (e.kind == EPI_RESID) {
          float* hp = e.h + (long)tok * e.h_ld + col;
          v += *hp;
          *hp = v;
        }
        red[t * (kTileN + 1) + f] = v;
        if (e.op) put_operand(e.op, (long)tok * e.op_ld + col, e.op_plane, v * (e.gain ? e.gain[col] : 1.f), e.op_f32);
      }
      epi_sync();
      if (e.ss_out) {
        const int warp = et >> 5, lane = et & 31;
        for (int t = warp; t < tc; t += kEpiThreads / 32) {
          float s = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float v = red[t * (kTileN + 1) + lane + 32 * q];
            s += v * v;
          }
          s = warp_sum(s);
          if (lane == 0) atomicAdd(e.ss_out + e.tok_base + tok0 + t, s);
        }
      }
    }
    epi_sync();
  }
}

}  // namespace dfl
