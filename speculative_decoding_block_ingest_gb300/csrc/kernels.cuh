// kernels.cuh -- host-side launch interface of the drafter kernels.
#pragma once
#include "dflash_internal.cuh"

namespace dfl {

// One weight-streaming projection: Y[tok][N] = X[tok][K] * W[N][K]^T with the
// fused epilogue e (swap-AB: W rows are tile rows, tokens are columns).
struct GemmArgs {
  const void* W;      // [N][K] in Geo::wtype
  int N, K;
  const void* X;      // operand [tok][K]: f32, or bf16 hi plane (+ lo plane at x_plane)
  int x_ld;
  long x_plane;
  int x_f32;
  Part p;
  int n_tiles;
  float* part;        // partial slots [(grid + n_tiles)][Mt][128]
  int* counters;      // [n_tiles], zero between calls
  EpiArgs e;
};

// Attention over the paged cache: per (seq, kv head, split) work item.
struct AttnArgs {
  const void* q;        // [Mt][Hq][d]  (kv dtype)
  const void* kpool;    // K pool base
  const void* vpool;    // V^T pool base
  int layer;
  const int* block_table;
  const RoundDesc* rd;
  float* part_o;        // [items][G*16][d]
  float* part_ml;       // [items][G*16][2]
  void* op;             // output operand [Mt][Hq*d] (hi/lo bf16 or f32)
  int op_ld;
  long op_plane;
  int op_f32;
  float scale;          // 1/sqrt(d)
  int* err;
  Geo g;
};

struct InitArgs {
  const float* src;     // noise [n_tok][H] (round) or taps [n_rows][n*H] (ingest)
  int n_rows, width;
  float* h;             // round: residual stream [Mt][H]
  float* ss0;           // round: ss of layer-0 input norm; ingest: null
  const float* gain;    // round: layer-0 input_ln
  void* op;             // operand output
  int op_ld;
  long op_plane;
  int op_f32;
  float* zero_ptr;      // floats to clear
  int zero_n;
  void* desc_dst;       // device descriptor
  int desc_bytes;
  int* block_table;
  Geo g;
};

void launch_gemm_simt(const GemmArgs& a, cudaStream_t s);
void launch_gemm_tc(const GemmArgs& a, const void* tmap_w, const void* tmap_x, cudaStream_t s);
void launch_attention_simt(const AttnArgs& a, int n_items, cudaStream_t s);
void launch_attn_combine(const AttnArgs& a, int n_tok, cudaStream_t s);
void launch_init(const InitArgs& a, const InitBlob& blob, cudaStream_t s);
void launch_final_norm(const float* h, const float* ss, const float* gain, float* out, int n_tok,
                       const Geo& g, cudaStream_t s);
void launch_kv_read(const Geo& g, const void* kpool, const void* vpool, const int* block_table,
                    int slot, int layer, int row0, int nrows, float* k_out, float* v_out,
                    cudaStream_t s);

}  // namespace dfl
