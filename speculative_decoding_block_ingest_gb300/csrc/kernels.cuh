// kernels.cuh -- host-side launch interface of the drafter kernels.
#pragma once
#include <utility>

#include "dflash_internal.cuh"

namespace dfl {

// Where a projection's result goes.
enum OMode {
  O_TILE = 0,     // stream-K ticket; the last arriver runs the tile epilogue EpiArgs::kind
  O_RED = 1       // every contributor red.adds into a token-major destination [tok][ld]
};

// One weight-streaming projection: Y[tok][N] = X[tok][K] * W[N][K]^T
// (swap-AB: W rows are tile rows, tokens are columns).
struct GemmArgs {
  const void* W;      // [N][K]: f32 rows, 16 KB bf16 blocks, or 8 KB e4m3 units (w8)
  int w8;             // tensor-core path: W is e4m3 codes (per-row scales in e.wscale)
  int N, K;
  const void* X;      // operand [tok][K]: f32, or bf16 hi plane (+ lo plane at x_plane)
  int x_ld;
  long x_plane;
  int x_f32;
  int omode;
  float* dst;         // O_RED: destination [tok][dst_ld]
  int dst_ld;
  Part p;
  int n_tiles;
  float* acc;         // O_TILE accumulators [n_tiles][128][nt], zero between calls
  int* counters;      // [n_tiles], zero between calls
  unsigned long long* trace;   // optional per-CTA timestamps [grid][kTraceWords], or null
  EpiArgs e;
};

// The small element-wise steps between the round's projections.
struct FinishArgs {
  int n_tok;
  int layer;
  const float* h;         // prep_norm: residual stream [Mt][H]
  const float* gain;      // prep_norm: RMSNorm gain [H]
  float* acc;             // qk_finish: QKV accumulator [Mt][qkv_n]; swiglu: gate/up [Mt][2I]
  void* op;               // prep_norm / swiglu: operand planes
  long op_plane;
  int op_kind;             // operand kind (OpKind)
  const float* qn;        // qk_finish: head-norm gains of this layer
  const float* kn;
  const float2* rope_cs;  // per token [d/2] (cos, sin) x mscale
  const int* dest;        // per token page*64 + offset of its (transient) K/V row
  void* q_out;            // [Mt][Hq][d]
  void* kpool;
  void* vpool;
  float* u_out;           // prep_norm: also the normed rows in f32 [Mt][H] (DFlash2 conv input), or null
  unsigned long long* trace;   // optional per-CTA entry / exit stamps, or null
  Geo g;
};

// A projection whose CTAs own whole 128-row tiles over the full K
// (proj_fused.cu): operand RMSNorm(h) x gain built in the kernel, the
// element-wise step after the projection in its epilogue.
enum OwnEpi { OWN_SWIGLU = 0 };
struct OwnArgs {
  const uint8_t* W;       // 16 KB weight blocks [tile][kb]
  int n_tiles, kb;        // tiles (one CTA each), 64-column units per tile
  int n_tok;
  const float* gain;      // RMSNorm gain [K]
  const float* wscale;    // per weight row scale (fp8), or null
  int epi;                // OwnEpi
  void* out;              // OWN_SWIGLU: the down projection's hi/lo bf16 operand planes
  int out_ld;
  long out_plane;
  unsigned long long* trace;
  int* err;
  Geo g;
};

// DFlash2 grouped dynamic causal conv of one sublayer over the block rows
// (16 per sequence, token t = 16 s + i; row i = 0 has no predecessor).
struct ConvArgs {
  int n_tok, groups;
  int half;               // 0: prepare (sublayer input -> operand planes); 1: finish (output -> residual add)
  const float* src;       // prepare: normed input u [Mt][H]; finish: sublayer output y [Mt][H]
  const float* base;      // [2][H][2] of this sublayer (tap 0 previous row, tap 1 this row)
  const float* dyn;       // [Mt][dyn_ld]: coefficients (half, group, tap) of this sublayer
  int dyn_ld;
  void* op;               // prepare: operand planes of the sublayer's first projection
  long op_plane;
  int op_kind;             // operand kind (OpKind)
  float* h;               // finish: residual stream [Mt][H]
  float* zero0;           // prepare: buffers the next projections red.add into, cleared here
  long zero0_n;
  float* zero1;
  long zero1_n;
  unsigned long long* trace;   // optional per-CTA entry / exit stamps, or null
  Geo g;
};

// Attention over the paged cache: per (seq, kv head, split) work item.
struct AttnArgs {
  const void* q;        // [Mt][Hq][d]  (kv dtype): normed, roped queries
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
  int op_kind;             // operand kind (OpKind)
  float scale_log2;     // log2(e)/sqrt(d): scores and the saved max are in log2 units
  int comb_wpr;         // merge: warps per merged row (attn_combine_wpr of the largest split count)
  int comb_max_split;   // merge: the largest split count of a row
  unsigned long long* trace;   // optional per-CTA timestamps [items][kTraceWords], or null
  int* err;
  Geo g;
};

struct InitArgs {
  const float* src;     // noise [n_tok][H] (round) or taps [n_rows][n*H] (ingest)
  int n_rows, width;
  float* h;             // round: residual stream [Mt][H] (then no operand is written)
  void* op;             // ingest: operand output
  int op_ld;
  long op_plane;
  int op_kind;             // operand kind (OpKind)
  float* zero_ptr;      // floats to clear
  int zero_n;
  void* desc_dst;       // device descriptor
  int cp_off[4], cp_len[4];   // word ranges of the descriptor that are used
                              // (head, positions, destinations, launch order)
  int* block_table;
  const double* inv_freq;   // RoPE inverse frequencies [d/2] (f64)
  float2* rope_cs;          // out: per row [d/2] (cos, sin) x mscale
  int is_round;             // positions come from blob.round.pos (else blob.ingest.row_pos)
  unsigned long long* trace;   // optional per-CTA entry / exit stamps, or null
  Geo g;
};

// Launch with programmatic stream serialization: the kernel may become
// resident while its predecessor drains; every kernel of the library calls
// griddepcontrol.wait before touching data a predecessor writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

void launch_gemm_simt(const GemmArgs& a, cudaStream_t s);
// tmap_h: the residual stream h [Mt][H] f32 with boxes of [nt rows][64 cols]
// (nt = the call's tokens rounded up to 16; 16 or 32).
cudaError_t launch_proj_own(const OwnArgs& a, const void* tmap_h, cudaStream_t s);
// Tensor-core projection: a.W is the weight in 16 KB blocks (see weights.cu).
void launch_gemm_tc(const GemmArgs& a, const void* tmap_x, cudaStream_t s);
// Token-tiled projection (gemm_tt.cu): bf16 or e4m3 weights, red.add results,
// more than 64 token rows, N a multiple of 256.  Units = gemm_tt_units; the
// operand map is the 128-row-box one.
bool gemm_tt_fits(const GemmArgs& a);
int gemm_tt_units(const GemmArgs& a);
void launch_gemm_tt(const GemmArgs& a, const void* tmap_x_tall, cudaStream_t s);
void launch_repack(void* dst, int K, const void* src, int n_rows, int chunk, int stride, int base, cudaStream_t s);
void launch_repack_e4m3(void* dst, int K, const void* src, int n_rows, int chunk, int stride, int base,
                        cudaStream_t s);

// Fixed device region of dflash_forward_full_static (static_full.cu).
constexpr size_t kFixedKvBytes = size_t(16) << 20;
constexpr int kFixedMaxDevices = 64;
cudaError_t fixed_kv_region(void** base, uint64_t user, bool* fresh);

// One bounded wait on a barrier nothing arrives on: records DERR_TIMEOUT in
// *err after limit_ns (selftest.cu).
void launch_selftest_wait(int* err, unsigned long long limit_ns, cudaStream_t s);
void launch_attention_simt(const AttnArgs& a, int n_items, cudaStream_t s);
void launch_attention_tc(const AttnArgs& a, int n_items, const void* tmq, const void* tmk, const void* tmv,
                         cudaStream_t s);
// Same over an e4m3 cache (head dim 128): tmq / tmk / tmv are the byte maps of
// the e4m3 queries, K pages and V^T pages.
void launch_attention_tc8(const AttnArgs& a, int n_items, const void* tmq, const void* tmk, const void* tmv,
                          cudaStream_t s);
void launch_prep_norm(const FinishArgs& f, cudaStream_t s);
void launch_qk_finish(const FinishArgs& f, int n_sm, cudaStream_t s);
void launch_swiglu(const FinishArgs& f, int n_sm, cudaStream_t s);
void launch_conv(const ConvArgs& c, int n_sm, cudaStream_t s);
void launch_attn_combine(const AttnArgs& a, int n_tok, cudaStream_t s);
// CTAs of the element-wise launches (trace regions are sized by them).
int prep_norm_grid(const FinishArgs& f);
int qk_finish_grid(const FinishArgs& f, int n_sm);
int swiglu_grid(const FinishArgs& f, int n_sm);
int conv_grid(const ConvArgs& c, int n_sm);
int attn_combine_grid(const AttnArgs& a, int n_tok);
int attn_combine_wpr(int max_split);
int init_grid(const InitArgs& a);
void launch_init(const InitArgs& a, const InitBlob& blob, cudaStream_t s);
const void* init_kernel_entry();       // kernel function addresses, to find
const void* final_norm_kernel_entry(); // their nodes in a captured graph
void launch_final_norm(const float* h, const float* gain, float* out, int n_tok, const Geo& g,
                       unsigned long long* trace, cudaStream_t s);
void launch_to_operand(const float* src, int n_rows, int width, void* op, long plane, cudaStream_t s);
void launch_argmax(const float* logits, int n_rows, int V, int32_t* tokens, cudaStream_t s);
void launch_kv_read(const Geo& g, const void* kpool, const void* vpool, const int* block_table,
                    int slot, int layer, int row0, int nrows, float* k_out, float* v_out,
                    cudaStream_t s);

}  // namespace dfl
