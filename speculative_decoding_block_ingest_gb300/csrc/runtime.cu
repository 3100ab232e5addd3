// runtime.cu -- host runtime and C ABI of the drafter round (include/dflash.h).
//
// The handle owns no device memory: everything lives in the caller's
// workspace, carved here.  Host-side state is the per-sequence page lists
// (one block table shared by all layers, spark_model::layers::dflash_head
// DflashProposerState), committed lengths, and the free-page pool.  Each call
// validates its arguments, then passes the per-call descriptor (positions,
// destination rows, new page-table entries) to its first kernel as a kernel
// parameter, so no host-to-device copy and no host synchronisation happen on
// the round's path.
#include <algorithm>
#include <functional>
#include <queue>
#include <atomic>
#include <cstdlib>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/dflash.h"
#include "kernels.cuh"

using namespace dfl;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

struct CudaError {
  std::string what;
};

void ck(cudaError_t e, const char* what) {
  if (e != cudaSuccess) throw CudaError{std::string(what) + ": " + cudaGetErrorString(e)};
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes per stored weight element: f32 rows, bf16 blocks of 16 KB, e4m3
// units of 8 KB (widened to f16 in shared memory by the projection).
int esize_w(int wtype) { return wtype == DFLASH_F32 ? 4 : (wtype == DFLASH_FP8_E4M3 ? 1 : 2); }

// Element type of the projections' operand planes for these weights.
int op_kind_of(int wtype) { return wtype == DFLASH_F32 ? OPK_F32 : (wtype == DFLASH_FP8_E4M3 ? OPK_F16 : OPK_BF16); }
int esize_kv(int kvtype) { return kvtype == DFLASH_F32 ? 4 : (kvtype == DFLASH_FP8_E4M3 ? 1 : 2); }

// Workspace carve-up, computed identically by dflash_workspace_bytes and dflash_create.
struct Layout {
  size_t fc, qkv, o, gu, down, kvall;                   // weights
  size_t s_fc, s_qkv, s_o, s_gu, s_down, s_kvall;       // fp8 row scales
  size_t hn, fn, in_ln, post_ln, qn, kn;                // norm gains
  size_t kpool, vpool, btab, inv_freq;
  size_t h, op_h, op_taps, op_o, op_a, q, qkv_acc, gu_acc, ss;
  size_t gacc, rope_cs, counters, apart_o, apart_ml, rdesc, idesc, err;
  size_t cbase, cdyn, s_cdyn, cu, cy, cdyn_a, cdyn_m;   // DFlash2 conv: weights, u / y rows, coefficients
  int conv_n;                                           // rows of a padded dynamic projection
  size_t total;
  int Mt, pps, max_tiles, grid_max, items_cap, n_sites;
};

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

// Attention work items a round's scratch holds: two waves of the SMs plus
// one item per kv head and sequence of the widest round.
int items_capacity(const dflash_config& c, int n_sm) {
  return std::min(2 * n_sm + c.n_kv_heads * c.max_batch, kMaxItems);
}

Layout make_layout(const dflash_config& c, int n_sm) {
  Layout Lo{};
  const size_t ew = esize_w(c.weight_dtype), ek = esize_kv(c.kv_dtype);
  const size_t L = c.n_layers, H = c.hidden, d = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads;
  const size_t I = c.intermediate, nH = (size_t)c.n_taps * H;
  const size_t qkv_n = (Hq + 2 * Hkv) * d, kv_n = 2 * Hkv * d;
  Lo.Mt = (int)align_up(std::max<size_t>((size_t)c.max_batch * kBlock, (size_t)c.max_ingest_rows), 16);
  Lo.pps = (c.max_seq_len + kPage - 1) / kPage;
  Lo.max_tiles = (int)std::max({qkv_n, H, 2 * I, L * kv_n}) / kTileN;
  Lo.grid_max = 2 * n_sm;
  Lo.n_sites = 2 + 4 * (int)L;
  const size_t G = Hq / Hkv, R = G * kBlock;
  Lo.items_cap = items_capacity(c, n_sm);
  const size_t Mt = Lo.Mt;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 1024);
    return at;
  };
  Lo.fc = take(H * nH * ew);
  Lo.qkv = take(L * qkv_n * H * ew);
  Lo.o = take(L * H * Hq * d * ew);
  Lo.gu = take(L * 2 * I * H * ew);
  Lo.down = take(L * H * I * ew);
  Lo.kvall = take(L * kv_n * H * ew);
  const bool fp8 = c.weight_dtype == DFLASH_FP8_E4M3;
  Lo.s_fc = take(fp8 ? H * 4 : 0);
  Lo.s_qkv = take(fp8 ? L * qkv_n * 4 : 0);
  Lo.s_o = take(fp8 ? L * H * 4 : 0);
  Lo.s_gu = take(fp8 ? L * 2 * I * 4 : 0);
  Lo.s_down = take(fp8 ? L * H * 4 : 0);
  Lo.s_kvall = take(fp8 ? L * kv_n * 4 : 0);
  Lo.hn = take(H * 4);
  Lo.fn = take(H * 4);
  Lo.in_ln = take(L * H * 4);
  Lo.post_ln = take(L * H * 4);
  Lo.qn = take(L * d * 4);
  Lo.kn = take(L * d * 4);
  // e4m3 pools carry their per-row scales after the codes
  const size_t kv_scales = c.kv_dtype == DFLASH_FP8_E4M3 ? L * (size_t)c.max_pages * Hkv * kPage * 4 : 0;
  Lo.kpool = take(L * (size_t)c.max_pages * Hkv * kPage * d * ek + kv_scales);
  Lo.vpool = take(L * (size_t)c.max_pages * Hkv * kPage * d * ek + kv_scales);
  Lo.btab = take((size_t)(c.max_seqs + 1) * Lo.pps * 4);
  Lo.inv_freq = take(d / 2 * 8);
  Lo.h = take(Mt * H * 4);
  Lo.op_h = take(Mt * H * 4);
  Lo.op_taps = take(Mt * nH * 4);
  Lo.op_o = take(Mt * Hq * d * 4);
  Lo.op_a = take(Mt * I * 4);
  Lo.q = take(Mt * Hq * d * 4);
  Lo.qkv_acc = take(Mt * qkv_n * 4);
  Lo.gu_acc = take(Mt * 2 * I * 4);
  Lo.ss = take((2 * L + 2) * Mt * 4);   // [2L+1]: ingest feature sums of squares
  Lo.gacc = take((size_t)Lo.max_tiles * kTileN * kPassTok * 4);
  Lo.rope_cs = take(Mt * d / 2 * 8);
  Lo.counters = take((size_t)Lo.n_sites * Lo.max_tiles * 4);
  Lo.apart_o = take((size_t)Lo.items_cap * R * d * 4);
  Lo.apart_ml = take((size_t)Lo.items_cap * R * 2 * 4);
  // DFlash2 conv: base kernels [L][2 sublayers][2][H][2], dynamic
  // projections [L][2][conv_n][H] (rows past 4 Gc zero), normed input and
  // sublayer output rows, coefficients of the two sublayers
  const size_t Gc = c.conv_groups;
  Lo.conv_n = Gc ? (int)align_up(4 * Gc, kTileN) : 0;
  Lo.cbase = take(Gc ? L * 2 * 2 * H * 2 * 4 : 0);
  Lo.cdyn = take(L * 2 * (size_t)Lo.conv_n * H * ew);
  Lo.s_cdyn = take(fp8 ? L * 2 * (size_t)Lo.conv_n * 4 : 0);
  Lo.cu = take(Gc ? Mt * H * 4 : 0);
  Lo.cy = take(Gc ? Mt * H * 4 : 0);
  Lo.cdyn_a = take(Mt * (size_t)Lo.conv_n * 4);
  Lo.cdyn_m = take(Mt * (size_t)Lo.conv_n * 4);
  Lo.rdesc = take(sizeof(RoundDesc));
  Lo.idesc = take(sizeof(IngestDesc));
  Lo.err = take(256);
  Lo.total = off;
  return Lo;
}

int validate_config(const dflash_config* c) {
  if (!c) return fail(DFLASH_ERR_INVALID_ARG, "config is null");
  if (c->n_layers < 1 || c->hidden < 128 || c->n_heads < 1 || c->n_kv_heads < 1 || c->intermediate < 64 ||
      c->n_taps < 1)
    return fail(DFLASH_ERR_INVALID_ARG, "non-positive dimension in config");
  if (c->hidden > kMaxHidden) return fail(DFLASH_ERR_UNSUPPORTED, "hidden must be at most %d", kMaxHidden);
  if (c->block != kBlock) return fail(DFLASH_ERR_UNSUPPORTED, "block must be 16 (got %d)", c->block);
  if (c->page_size != kPage) return fail(DFLASH_ERR_UNSUPPORTED, "page_size must be 64 (got %d)", c->page_size);
  if (c->head_dim != 64 && c->head_dim != 128) return fail(DFLASH_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->n_heads % c->n_kv_heads) return fail(DFLASH_ERR_INVALID_ARG, "n_heads %% n_kv_heads != 0");
  if (c->n_heads / c->n_kv_heads > 8) return fail(DFLASH_ERR_UNSUPPORTED, "more than 8 q heads per kv head");
  const long qkv_n = (long)(c->n_heads + 2 * c->n_kv_heads) * c->head_dim;
  if (c->hidden % kTileN || qkv_n % kTileN || (2L * c->n_kv_heads * c->head_dim * c->n_layers) % kTileN ||
      c->intermediate % 64 || ((long)c->n_heads * c->head_dim) % kTileK)
    return fail(DFLASH_ERR_UNSUPPORTED, "projection sizes must be multiples of 128 rows / 64 columns");
  if (c->weight_dtype < DFLASH_F32 || c->weight_dtype > DFLASH_FP8_E4M3) return fail(DFLASH_ERR_INVALID_ARG, "weight_dtype");
  if (c->kv_dtype != DFLASH_F32 && c->kv_dtype != DFLASH_BF16 && c->kv_dtype != DFLASH_FP8_E4M3)
    return fail(DFLASH_ERR_INVALID_ARG, "kv_dtype");
  if (c->weight_dtype == DFLASH_F32 && c->kv_dtype != DFLASH_F32)
    return fail(DFLASH_ERR_UNSUPPORTED, "f32 weights need an f32 KV cache");
  if (c->weight_dtype != DFLASH_F32 && c->kv_dtype == DFLASH_F32)
    return fail(DFLASH_ERR_UNSUPPORTED, "bf16/fp8 weights need a bf16 or e4m3 KV cache");
  if (c->kv_dtype == DFLASH_FP8_E4M3 && c->head_dim != 128)
    return fail(DFLASH_ERR_UNSUPPORTED, "an e4m3 KV cache needs head_dim 128");
  if (c->rope_type != DFLASH_ROPE_PLAIN && c->rope_type != DFLASH_ROPE_YARN) return fail(DFLASH_ERR_INVALID_ARG, "rope_type");
  if (!(c->rope_theta > 1.0)) return fail(DFLASH_ERR_INVALID_ARG, "rope_theta must be > 1");
  if (c->rope_type == DFLASH_ROPE_YARN &&
      (!(c->yarn_factor >= 1.0) || c->yarn_original_max_pos < 1 || !(c->yarn_beta_fast > 0) || !(c->yarn_beta_slow > 0)))
    return fail(DFLASH_ERR_INVALID_ARG, "bad YaRN parameters");
  if (!(c->rms_eps > 0)) return fail(DFLASH_ERR_INVALID_ARG, "rms_eps must be > 0");
  if (c->max_seqs < 1 || c->max_pages < 1 || c->max_seq_len < kBlock + 1)
    return fail(DFLASH_ERR_INVALID_ARG, "capacity fields must be positive");
  if (c->max_batch < 1 || c->max_batch > kMaxBatch) return fail(DFLASH_ERR_INVALID_ARG, "max_batch must be 1..64");
  if ((long)c->n_kv_heads * c->max_batch > kMaxItems)
    return fail(DFLASH_ERR_INVALID_ARG, "n_kv_heads x max_batch must be at most %d", kMaxItems);
  if (c->max_ingest_rows < 1 || c->max_ingest_rows > kMaxIngestRows)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ingest_rows must be 1..512");
  if (c->conv_groups < 0 || c->conv_groups > kMaxConvGroups ||
      (c->conv_groups > 0 && (c->hidden % c->conv_groups || (c->hidden / c->conv_groups) % 4)))
    return fail(DFLASH_ERR_INVALID_ARG, "conv_groups must be 0, or divide hidden into groups of a multiple of 4 (at most %d)",
                kMaxConvGroups);
  return DFLASH_OK;
}

// RoPE inverse frequencies: plain theta^(-2j/d), or the YaRN remap
// theta^(-2j/d)/ff[j] of the DflashDraft page (item rope_yarn), with ff the
// by-dimension blend between 1 and the factor over the correction range.
void rope_table(const dflash_config& c, std::vector<double>& inv, float& mscale) {
  const int d = c.head_dim, half = d / 2;
  inv.resize(half);
  for (int j = 0; j < half; ++j) inv[j] = std::pow(c.rope_theta, -2.0 * j / d);
  mscale = 1.f;
  if (c.rope_type != DFLASH_ROPE_YARN) return;
  auto corr = [&](double turns) {
    return d * std::log(c.yarn_original_max_pos / (turns * 2.0 * M_PI)) / (2.0 * std::log(c.rope_theta));
  };
  double lo = std::max(std::floor(corr(c.yarn_beta_fast)), 0.0);
  double hi = std::min(std::ceil(corr(c.yarn_beta_slow)), (double)(d - 1));
  if (lo == hi) hi += 0.001;
  for (int j = 0; j < half; ++j) {
    double ramp = std::min(1.0, std::max(0.0, (j - lo) / (hi - lo)));
    double ff = 1.0 / ((1.0 - ramp) + ramp / c.yarn_factor);
    inv[j] /= ff;
  }
  mscale = (float)(0.1 * std::log(c.yarn_factor) + 1.0);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    ck(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q),
       "driver entry point cuTensorMapEncodeTiled");
    if (q != cudaDriverEntryPointSuccess || !p) throw CudaError{"cuTensorMapEncodeTiled unavailable"};
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 map over a row-major [rows][cols] matrix, box [box_rows][64] in
// the 128-byte swizzle (the layout the MMA descriptors expect).
CUtensorMap make_map_bf16(const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  CUtensorMap m;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) throw CudaError{"cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")"};
  return m;
}

// 2-D f32 map over a row-major [rows][cols] matrix, box [box_rows][64], no swizzle.
CUtensorMap make_map_f32(const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  CUtensorMap m;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) throw CudaError{"cuTensorMapEncodeTiled (f32) failed (" + std::to_string((int)r) + ")"};
  return m;
}

// 3-D bf16 map over [d2][d1][d0] (d0 innermost), box {64, b1, b2}, 128-byte swizzle.
CUtensorMap make_map_bf16_3d(const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1, uint32_t b2) {
  CUtensorMap m;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = tensor_map_encoder()(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) throw CudaError{"cuTensorMapEncodeTiled (3-D) failed (" + std::to_string((int)r) + ")"};
  return m;
}

// 2-D byte map over [rows][cols] (e4m3 codes), box [box_rows][box_cols].
CUtensorMap make_map_u8(const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                        CUtensorMapSwizzle swz) {
  CUtensorMap m;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) throw CudaError{"cuTensorMapEncodeTiled (u8) failed (" + std::to_string((int)r) + ")"};
  return m;
}

}  // namespace

struct dflash_handle {
  dflash_config cfg;
  Layout lo;
  char* ws;
  Geo g;
  int n_sm;
  std::vector<int64_t> len;               // committed rows per slot (slot max_seqs = internal)
  std::vector<std::vector<int>> pages;    // page ids per slot (in the current KV region); -1 = evicted
  // context window (dflash_set_ctx_cap): 0 = unbounded; per slot the first
  // position still kept and attended
  int64_t ctx_cap = 0;
  std::vector<int64_t> kstart;
  bool evicted_any = false;
  // A KV region: K and V^T pools of `max_pages` pages per layer, their
  // tensor maps and free list.  `pool` lives in the workspace; `fixed` is the
  // library's static device region used by dflash_forward_full_static.
  struct KvRegion {
    char* kpool = nullptr;
    char* vpool = nullptr;
    int max_pages = 0;
    CUtensorMap kmap, vmap;
    std::vector<int> free_pages;
  };
  KvRegion pool, fixed;
  KvRegion* kv = &pool;                   // region the enqueued kernels use
  cudaStream_t last_stream = nullptr;
  // measurement: kernel launches issued, and (when enabled) per-kind event pairs
  int64_t launches = 0;
  // tensor maps of the tensor-core projections' operands (per buffer)
  // operand maps: [0] boxes of 16 rows, [1] boxes of 128 rows (passes of >= 128 tokens)
  CUtensorMap xmap_taps[2], xmap_h[2], xmap_o[2], xmap_a[2];
  CUtensorMap hmap[2];                          // residual stream h (f32), boxes of 16 / 32 rows x 64 columns
  CUtensorMap qmap;                             // attention: q buffer (3-D)
  bool use_tc = false;    // tensor-core projections (bf16 weights)
  bool attn_tc = false;   // tensor-core attention (bf16 KV, any weights)
  bool prof_on = false;
  // replayable rounds: one instantiated graph per (sequences, attention
  // items, KV region); only the per-call init and final-norm nodes change
  struct RoundGraph {
    int n_seq = 0, n_items = 0;
    const void* region = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaGraphNode_t init_node = nullptr, norm_node = nullptr;
    cudaKernelNodeParams init_p{}, norm_p{};
    int64_t launches = 0;
    uint64_t used = 0;
  };
  std::vector<RoundGraph> graphs;
  uint64_t graph_clock = 0;
  bool attn_fp8 = false;        // e4m3 KV cache: attention on kind::f8f6f4 scores
  uint64_t uid = 0;             // process-unique handle id (static region ownership)
  int device = -1;              // the device current at create (its workspace, weights and static region)
  cudaStream_t cap_stream = nullptr;   // private stream the rounds are captured on
  struct Rec {
    int kind;
    cudaEvent_t a, b;
    double bytes;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> event_pool;
  // launch trace (per-CTA timestamps) into a caller buffer
  unsigned long long* trace_buf = nullptr;
  size_t trace_cap = 0, trace_used = 0;   // in u64 words
  struct TraceRec {
    int kind, grid;
    int64_t offset;
  };
  std::vector<TraceRec> trace_recs;
  std::vector<cudaGraphExec_t> traced_execs;   // traced rounds' graphs, kept until tracing stops
  template <class T>
  T* at(size_t off) { return reinterpret_cast<T*>(ws + off); }
};

namespace {

cudaEvent_t take_event(dflash_t* h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e;
  ck(cudaEventCreate(&e), "event create");
  return e;
}

// Brackets one kernel launch: counts it and, when profiling is on, records
// an event pair on the launch stream with the launch's algorithmic bytes.
struct Launch {
  dflash_t* h;
  cudaStream_t s;
  int idx = -1;
  Launch(dflash_t* h_, int kind, double bytes, cudaStream_t s_) : h(h_), s(s_) {
    ++h->launches;
    if (h->prof_on) {
      dflash_handle::Rec r{kind, take_event(h), take_event(h), bytes};
      ck(cudaEventRecord(r.a, s), "event record");
      h->recs.push_back(r);
      idx = (int)h->recs.size() - 1;
    }
  }
  ~Launch() {
    if (idx >= 0) cudaEventRecord(h->recs[idx].b, s);
  }
};

// Next free trace region for a launch of `grid` CTAs (null when tracing is off or full).
unsigned long long* trace_slot(dflash_t* h, int kind, int grid) {
  if (!h->trace_buf) return nullptr;
  const size_t words = (size_t)grid * kTraceWords;
  if (h->trace_used + words > h->trace_cap) return nullptr;
  unsigned long long* p = h->trace_buf + h->trace_used;
  h->trace_recs.push_back({kind, grid, (int64_t)h->trace_used});
  h->trace_used += words;
  return p;
}

// Reserve pages so that slot covers `rows` rows; records block-table entries.
bool ensure_pages(dflash_t* h, int slot, int64_t rows, InitBlob& blob, std::vector<int>& taken) {
  const int need = (int)((rows + kPage - 1) / kPage);
  auto& pl = h->pages[slot];
  while ((int)pl.size() < need) {
    auto& fl = h->kv->free_pages;
    if (fl.empty() || blob.n_pt >= kMaxPtUpdates) return false;
    const int page = fl.back();
    fl.pop_back();
    taken.push_back(slot);
    blob.pt_idx[blob.n_pt] = slot * h->lo.pps + (int)pl.size();
    blob.pt_page[blob.n_pt] = page;
    ++blob.n_pt;
    pl.push_back(page);
  }
  return true;
}

// Undo ensure_pages for a failed call.
void rollback_pages(dflash_t* h, const InitBlob& blob, const std::vector<int>& taken) {
  for (int i = (int)taken.size() - 1; i >= 0; --i) {
    auto& pl = h->pages[taken[i]];
    h->kv->free_pages.push_back(pl.back());
    pl.pop_back();
  }
  (void)blob;
}

// CTAs of a tensor-core projection pass.  At 16 tokens the tensor-core path
// of one SM moves about 90 GB/s of weights (the MMA issue rate, not memory,
// bounds it), so a projection takes every SM to stream HBM at full rate.
#ifndef DFLASH_GEMM_GRID
#define DFLASH_GEMM_GRID 152
#endif
int proj_grid(const dflash_t* h, int n_tok) {
  return n_tok <= 64 ? std::min(h->n_sm, DFLASH_GEMM_GRID) : h->n_sm;
}

EpiArgs base_epi(dflash_t* h) {
  EpiArgs e{};
  e.g = h->g;
  e.rope_cs = h->at<float2>(h->lo.rope_cs);
  e.kpool = h->kv->kpool;
  e.vpool = h->kv->vpool;
  e.err = h->at<int>(h->lo.err);
  e.op_kind = op_kind_of(h->cfg.weight_dtype);
  return e;
}

// One projection call: its operand, where its result goes, and (for the
// ingest's projections) the tile epilogue.
struct GemmSpec {
  int site;                     // weight map and counter block
  const void* W;
  const float* wscale;          // per-row scales of e4m3 weights (8 KB units); nullptr: bf16 / f32 weights
  int N, K;
  const void* X = nullptr;      // operand planes (bf16 or f16 hi/lo, or f32)
  const CUtensorMap* xmap = nullptr;   // [short, tall] operand maps
  int omode = O_TILE;
  float* dst = nullptr;         // O_RED destination [tok][dst_ld]
  int dst_ld = 0;
  int grid = 0;                 // CTAs of a tensor-core pass (0: proj_grid)
  EpiArgs e;
};

// Passes of <= 256 token columns; tensor cores for bf16 and e4m3 weights,
// CUDA cores for f32 weights.
void run_gemm(dflash_t* h, const GemmSpec& sp, cudaStream_t s) {
  const Geo& g = h->g;
  const int n_all = sp.e.n_tok;
  if (h->use_tc && 2 * h->lo.Mt >= 256) {
    // more than 64 rows into a red.add destination: one token-tiled launch
    // over every row (weights streamed once)
    GemmArgs a{};
    a.W = sp.W;
    a.w8 = sp.wscale != nullptr;
    a.N = sp.N;
    a.K = sp.K;
    a.omode = sp.omode;
    a.dst = sp.dst;
    a.dst_ld = sp.dst_ld;
    a.e = sp.e;
    a.e.wscale = sp.wscale;
    a.e.tok_base = 0;
    a.e.n_tok = n_all;
    if (gemm_tt_fits(a)) {
      a.n_tiles = sp.N / kTileN;
      a.p.kb = sp.K / kTileK;
      a.p.units = gemm_tt_units(a);
      a.p.grid = std::min(a.p.units, h->n_sm);
      const double bytes = (double)sp.N * sp.K * (a.w8 ? 1 : 2) + (a.w8 ? sp.N * 4.0 : 0.0) + (double)n_all * sp.K * 4 +
                           (double)n_all * sp.N * 4;
      Launch L(h, DFLASH_KERNEL_GEMM, bytes, s);
      a.trace = trace_slot(h, DFLASH_KERNEL_GEMM, a.p.grid);
      launch_gemm_tt(a, &sp.xmap[1], s);
      ck(cudaGetLastError(), "token-tiled gemm launch");
      return;
    }
  }
  for (int base = 0; base < n_all; base += kPassTok) {
    GemmArgs a{};
    a.W = sp.W;
    a.w8 = sp.wscale != nullptr;
    a.N = sp.N;
    a.K = sp.K;
    a.X = sp.X;
    a.x_ld = sp.K;
    a.x_plane = (long)h->lo.Mt * sp.K;
    a.x_f32 = h->cfg.weight_dtype == DFLASH_F32;
    a.omode = sp.omode;
    a.dst = sp.dst;
    a.dst_ld = sp.dst_ld;
    a.n_tiles = sp.N / kTileN;
    a.p.kb = sp.K / kTileK;
    a.p.units = a.n_tiles * a.p.kb;
    a.p.grid = std::min(a.p.units, !h->use_tc ? h->lo.grid_max
                                              : sp.grid > 0 ? sp.grid : proj_grid(h, std::min(kPassTok, n_all - base)));
    a.acc = h->at<float>(h->lo.gacc);
    a.counters = h->at<int>(h->lo.counters) + (size_t)sp.site * h->lo.max_tiles;
    a.e = sp.e;
    a.e.wscale = sp.wscale;
    a.e.tok_base = base;
    a.e.n_tok = std::min(kPassTok, n_all - base);
    const double nt = a.e.n_tok;
    // algorithmic bytes: weights (+ scales), the operand once, the result once
    double x_b = nt * sp.K * 4;
    double out_b;
    if (sp.omode == O_RED) out_b = nt * sp.N * 4;
    else if (sp.e.kind == EPI_FC) out_b = nt * sp.N * 4;
    else out_b = nt * sp.N * (g.kvtype == KV_F32 ? 4 : (g.kvtype == KV_FP8 ? 1.0 + 4.0 / g.d : 2));
    const double ew = a.w8 ? 1.0 : (h->cfg.weight_dtype == DFLASH_F32 ? 4.0 : 2.0);
    const double bytes = (double)sp.N * sp.K * ew + (sp.wscale ? sp.N * 4.0 : 0.0) + x_b + out_b;
    Launch L(h, DFLASH_KERNEL_GEMM, bytes, s);
    a.trace = h->use_tc ? trace_slot(h, DFLASH_KERNEL_GEMM, a.p.grid) : nullptr;
    if (h->use_tc) launch_gemm_tc(a, sp.xmap, s);
    else launch_gemm_simt(a, s);
  }
  ck(cudaGetLastError(), "gemm launch");
}

size_t wbytes(dflash_t* h) { return esize_w(h->cfg.weight_dtype); }

// Ingest rows already validated and paged; blob.ingest filled.
void enqueue_ingest(dflash_t* h, const InitBlob& blob, const float* taps, cudaStream_t s) {
  const Geo& g = h->g;
  const int n_rows = blob.ingest.n_rows;
  const int width = g.n * g.H;
  InitArgs ia{};
  ia.src = taps;
  ia.n_rows = n_rows;
  ia.width = width;
  ia.h = nullptr;
  ia.op = h->at<void>(h->lo.op_taps);
  ia.op_ld = width;
  ia.op_plane = (long)h->lo.Mt * width;
  ia.op_kind = op_kind_of(h->cfg.weight_dtype);
  float* ss_feat = h->at<float>(h->lo.ss) + (size_t)(2 * g.L + 1) * h->lo.Mt;
  ia.zero_ptr = ss_feat;
  ia.zero_n = n_rows;
  ia.desc_dst = h->at<void>(h->lo.idesc);
  ia.cp_off[0] = 0;
  ia.cp_len[0] = (int)(offsetof(IngestDesc, row_pos) / 4);
  ia.cp_off[1] = (int)(offsetof(IngestDesc, row_pos) / 4);
  ia.cp_len[1] = n_rows;
  ia.cp_off[2] = (int)(offsetof(IngestDesc, row_dest) / 4);
  ia.cp_len[2] = n_rows;
  ia.block_table = h->at<int>(h->lo.btab);
  ia.inv_freq = h->at<double>(h->lo.inv_freq);
  ia.rope_cs = h->at<float2>(h->lo.rope_cs);
  ia.is_round = 0;
  ia.g = g;
  {
    Launch L(h, DFLASH_KERNEL_INIT, (double)n_rows * width * 8, s);
    ia.trace = trace_slot(h, DFLASH_KERNEL_INIT, init_grid(ia));
    launch_init(ia, blob, s);
  }
  ck(cudaGetLastError(), "ingest init launch");

  // fc over the taps; epilogue: feats operand (c * hidden_norm) + sum c^2
  const bool fp8 = h->cfg.weight_dtype == DFLASH_FP8_E4M3;
  GemmSpec fc;
  fc.site = 0;
  fc.W = h->at<void>(h->lo.fc);
  fc.wscale = fp8 ? h->at<float>(h->lo.s_fc) : nullptr;
  fc.N = g.H;
  fc.K = width;
  fc.X = h->at<void>(h->lo.op_taps);
  fc.xmap = h->xmap_taps;
  fc.e = base_epi(h);
  fc.e.kind = EPI_FC;
  fc.e.n_tok = n_rows;
  fc.e.ss_out = ss_feat;
  fc.e.gain = h->at<float>(h->lo.hn);
  fc.e.op = h->at<void>(h->lo.op_h);
  fc.e.op_ld = g.H;
  fc.e.op_plane = (long)h->lo.Mt * g.H;
  run_gemm(h, fc, s);

  // K/V of every layer in one projection; epilogue: hidden_norm scale,
  // k head-norm + RoPE, paged write.
  GemmSpec kv;
  kv.site = 1;
  kv.W = h->at<void>(h->lo.kvall);
  kv.wscale = fp8 ? h->at<float>(h->lo.s_kvall) : nullptr;
  kv.N = g.L * g.kv_n;
  kv.K = g.H;
  kv.X = h->at<void>(h->lo.op_h);
  kv.xmap = h->xmap_h;
  kv.e = base_epi(h);
  kv.e.kind = EPI_KV;
  kv.e.n_tok = n_rows;
  kv.e.ss_in = ss_feat;
  kv.e.kn = h->at<float>(h->lo.kn);
  kv.e.dest = h->at<IngestDesc>(h->lo.idesc)->row_dest;
  run_gemm(h, kv, s);
}

// Pages from the one holding each sequence's first attended key through its
// block rows.
static std::vector<long> attended_pages(const std::vector<int64_t>& lens, const int* kstart) {
  std::vector<long> pages(lens.size());
  for (size_t i = 0; i < lens.size(); ++i) pages[i] = (lens[i] + kBlock + kPage - 1) / kPage - kstart[i] / kPage;
  return pages;
}

// Finishing time of a round's attention items (pages each plus a fixed
// per-item cost of about two chunks), launched longest first, each CTA
// taking the SM that frees first among `slots`.
static long schedule_span(const std::vector<long>& pages, int Hkv, long sp, long slots, long item_cost,
                          std::vector<long>& scratch) {
  scratch.clear();
  for (long p : pages)
    for (long k0 = 0; k0 < p; k0 += sp) scratch.insert(scratch.end(), Hkv, std::min(sp, p - k0) + item_cost);
  std::stable_sort(scratch.begin(), scratch.end(), std::greater<long>());
  std::priority_queue<long, std::vector<long>, std::greater<long>> free_at;
  long span = 0;
  for (long c : scratch) {
    long t = 0;
    if ((long)free_at.size() >= slots) {
      t = free_at.top();
      free_at.pop();
    }
    free_at.push(t + c);
    span = std::max(span, t + c);
  }
  return span;
}

// What the attention plan depends on besides the sequences: kv heads, the
// item scratch, and how many items run at once.
struct AttnPlanCtx {
  int Hkv;
  long items_cap;
  long slots;
};

// Items run `slots` at a time: one per SM for the tensor-core kernels, beside
// a small round's projection when that leaves at least 32 SMs (so that the
// two kernels can be resident together), two per SM for the SIMT kernel.
static AttnPlanCtx attn_plan_ctx(int Hkv, long items_cap, int n_sm, bool attn_tc, int n_tok) {
  const long proj = n_tok <= 64 ? std::min(n_sm, DFLASH_GEMM_GRID) : n_sm;   // proj_grid
  const long beside = (long)n_sm - proj;
  AttnPlanCtx c;
  c.Hkv = Hkv;
  c.items_cap = items_cap;
  c.slots = attn_tc ? (n_tok <= 64 && beside >= 32 ? beside : (long)n_sm) : 2L * n_sm;
  return c;
}

static int choose_split_pages(const AttnPlanCtx& c, const std::vector<long>& pages) {
  long units = 0, longest = 1;
  for (long p : pages) {
    units += (long)c.Hkv * p;
    longest = std::max(longest, p);
  }
  // Items go to SMs as earlier ones finish (launched longest first), so
  // score a few split sizes by that schedule: the per-SM share of all pages
  // and its halves, thirds, ... (and the wave-count choice below).  Among
  // equal spans the larger split wins (fewer partials to merge).
  const long slots = c.slots;
  constexpr long kItemCost = 4;
  auto items_of = [&](long sp) {
    long items = 0;
    for (long p : pages) items += (long)c.Hkv * ((p + sp - 1) / sp);
    return items;
  };
  // the split minimising waves x (pages per item + the fixed cost), as if
  // items ran in lockstep waves
  long wave_sp = longest, best_wave = -1;
  for (long sp = 1; sp <= longest; ++sp) {
    const long items = items_of(sp);
    if (items > c.items_cap) continue;   // sp = longest always fits: Hkv items a sequence
    const long cost = (items + slots - 1) / slots * (sp + kItemCost);
    if (best_wave < 0 || cost <= best_wave) {
      wave_sp = sp;
      best_wave = cost;
    }
  }
  std::vector<long> cand = {wave_sp, longest};
  const long share = (units + slots - 1) / slots;
  for (long k = 1; k <= 8; ++k) cand.push_back(std::max(1L, (share + k - 1) / k));
  std::sort(cand.begin(), cand.end(), std::greater<long>());
  cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
  std::vector<long> scratch;
  long best = wave_sp, best_span = -1;
  for (long sp : cand) {
    if (sp > longest || items_of(sp) > c.items_cap) continue;
    const long span = schedule_span(pages, c.Hkv, sp, slots, kItemCost, scratch);
    if (best_span < 0 || span < best_span) {
      best = sp;
      best_span = span;
    }
  }
  return (int)best;
}

// The split size, each sequence's first item (item0[n_seq] = the item count)
// and, when the count fits kMaxItems, the launch order (CTA c runs item
// order[c]): items are (sequence, kv head, split) in that order, launched
// longest first, ties in item order, so short remainders fill in last.
static int plan_items(const AttnPlanCtx& c, const std::vector<long>& pages, int* item0, uint16_t* order) {
  const int sp = choose_split_pages(c, pages);
  std::vector<std::pair<long, int>> by_len;
  int items = 0;
  for (size_t s = 0; s < pages.size(); ++s) {
    item0[s] = items;
    const long n_split = (pages[s] + sp - 1) / sp;
    for (int kvh = 0; kvh < c.Hkv; ++kvh)
      for (long j = 0; j < n_split; ++j) by_len.push_back({std::min<long>(sp, pages[s] - j * sp), items++});
  }
  item0[pages.size()] = items;
  if (items <= kMaxItems) {
    std::stable_sort(by_len.begin(), by_len.end(),
                     [](const std::pair<long, int>& a, const std::pair<long, int>& b) { return a.first > b.first; });
    for (int k = 0; k < items; ++k) order[k] = (uint16_t)by_len[k].second;
  }
  return sp;
}

// Arguments of a round's init kernel (copied into the kernel's parameters).
InitArgs round_init_args(dflash_t* h, const RoundDesc& rd, const float* noise) {
  const int n_tok = rd.n_tok;
  InitArgs ia{};
  ia.src = noise;
  ia.n_rows = n_tok;
  ia.width = h->g.H;
  ia.h = h->at<float>(h->lo.h);
  ia.desc_dst = h->at<void>(h->lo.rdesc);
  ia.cp_off[0] = 0;
  ia.cp_len[0] = (int)(offsetof(RoundDesc, pos) / 4);
  ia.cp_off[1] = (int)(offsetof(RoundDesc, pos) / 4);
  ia.cp_len[1] = n_tok;
  ia.cp_off[2] = (int)(offsetof(RoundDesc, dest) / 4);
  ia.cp_len[2] = n_tok;
  ia.cp_off[3] = (int)(offsetof(RoundDesc, perm) / 4);
  ia.cp_len[3] = (rd.n_items + 1) / 2;   // two 16-bit entries a word
  ia.block_table = h->at<int>(h->lo.btab);
  ia.inv_freq = h->at<double>(h->lo.inv_freq);
  ia.rope_cs = h->at<float2>(h->lo.rope_cs);
  ia.is_round = 1;
  ia.g = h->g;
  if (h->cfg.conv_groups > 0) {
    // the first layer's attention coefficients are red.added from zero
    ia.zero_ptr = h->at<float>(h->lo.cdyn_a);
    ia.zero_n = n_tok * h->lo.conv_n;
  }
  return ia;
}

// The round: per layer
//   prep_norm(input_ln) -> QKV -> qk_finish -> attention -> combine -> O ->
//   prep_norm(post_ln) -> gate/up -> swiglu -> down.
// The projections only stream weights: their operands are prepared planes
// read by TMA, and their results are red.added into token-major
// accumulators (QKV, gate/up) or into the residual stream h (O, down).  The
// small element-wise steps run as wide kernels in between (finish.cu), all
// chained by programmatic dependent launch.
void enqueue_round(dflash_t* h, InitBlob& blob, const float* noise, float* out, cudaStream_t s) {
  const Geo& g = h->g;
  RoundDesc& rd = blob.round;
  const int n_tok = rd.n_tok;
  const size_t Mt = h->lo.Mt;
  const bool fp8 = h->cfg.weight_dtype == DFLASH_FP8_E4M3;
  const size_t ew = wbytes(h);
  float* hres = h->at<float>(h->lo.h);
  float* qkv_acc = h->at<float>(h->lo.qkv_acc);
  float* gu_acc = h->at<float>(h->lo.gu_acc);

  InitArgs ia = round_init_args(h, rd, noise);
  {
    Launch L(h, DFLASH_KERNEL_INIT, (double)n_tok * g.H * 8, s);
    ia.trace = trace_slot(h, DFLASH_KERNEL_INIT, init_grid(ia));
    launch_init(ia, blob, s);
  }
  ck(cudaGetLastError(), "round init launch");

  FinishArgs fb{};
  fb.n_tok = n_tok;
  fb.h = hres;
  fb.op_kind = op_kind_of(h->cfg.weight_dtype);
  fb.rope_cs = h->at<float2>(h->lo.rope_cs);
  fb.dest = h->at<RoundDesc>(h->lo.rdesc)->dest;
  fb.q_out = h->at<void>(h->lo.q);
  fb.kpool = h->kv->kpool;
  fb.vpool = h->kv->vpool;
  fb.g = g;
  // DFlash2: the grouped dynamic causal conv around each sublayer
  const int Gc = h->cfg.conv_groups, conv_n = h->lo.conv_n;
  float* cu = Gc ? h->at<float>(h->lo.cu) : nullptr;
  float* cy = Gc ? h->at<float>(h->lo.cy) : nullptr;
  float* dyn_sub[2] = {h->at<float>(h->lo.cdyn_a), h->at<float>(h->lo.cdyn_m)};
  // the MLP's norm, gate/up and SwiGLU as one tile-owning projection: tensor
  // cores, no DFlash2 conv around the sublayer, up to 32 block rows, a tile
  // per SM
  const bool fused_mlp = h->use_tc && !fp8 && !Gc && n_tok <= 32 && 2 * g.I / kTileN <= h->n_sm;
  auto prep_norm = [&](const float* gain) {
    FinishArgs f = fb;
    f.gain = gain;
    f.op = h->at<void>(h->lo.op_h);
    f.op_plane = (long)Mt * g.H;
    f.u_out = cu;
    Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * g.H * (Gc ? 12 : 8), s);
    f.trace = trace_slot(h, DFLASH_KERNEL_FINISH, prep_norm_grid(f));
    launch_prep_norm(f, s);
  };
  // prepare: the dynamic coefficients of sublayer `sub` (both halves) from
  // its normed input, then the input through half 0 into the operand planes;
  // clears the output rows and the other sublayer's coefficients, which the
  // next projections red.add into
  auto conv_prepare = [&](int l, int sub) {
    const size_t m = (size_t)l * 2 + sub;
    GemmSpec cd;
    cd.site = 2 + 4 * l;
    cd.W = h->at<char>(h->lo.cdyn) + m * conv_n * g.H * ew;
    cd.wscale = fp8 ? h->at<float>(h->lo.s_cdyn) + m * conv_n : nullptr;
    cd.N = conv_n;
    cd.K = g.H;
    cd.X = h->at<void>(h->lo.op_h);
    cd.xmap = h->xmap_h;
    cd.omode = O_RED;
    cd.dst = dyn_sub[sub];
    cd.dst_ld = conv_n;
    cd.e = base_epi(h);
    cd.e.n_tok = n_tok;
    run_gemm(h, cd, s);
    ConvArgs c{};
    c.n_tok = n_tok;
    c.groups = Gc;
    c.half = 0;
    c.src = cu;
    c.base = h->at<float>(h->lo.cbase) + m * 2 * g.H * 2;
    c.dyn = dyn_sub[sub];
    c.dyn_ld = conv_n;
    c.op = h->at<void>(h->lo.op_h);
    c.op_plane = (long)Mt * g.H;
    c.op_kind = op_kind_of(h->cfg.weight_dtype);
    c.zero0 = cy;
    c.zero0_n = (long)n_tok * g.H;
    c.zero1 = dyn_sub[sub ^ 1];
    c.zero1_n = (long)n_tok * conv_n;
    c.g = g;
    Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * g.H * 20, s);
    c.trace = trace_slot(h, DFLASH_KERNEL_FINISH, conv_grid(c, h->n_sm));
    launch_conv(c, h->n_sm, s);
    ck(cudaGetLastError(), "conv prepare launch");
  };
  // finish: the sublayer output through half 1, added into the residual
  auto conv_finish = [&](int l, int sub) {
    ConvArgs c{};
    c.n_tok = n_tok;
    c.groups = Gc;
    c.half = 1;
    c.src = cy;
    c.base = h->at<float>(h->lo.cbase) + ((size_t)l * 2 + sub) * 2 * g.H * 2;
    c.dyn = dyn_sub[sub];
    c.dyn_ld = conv_n;
    c.h = hres;
    c.g = g;
    Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * g.H * 16, s);
    c.trace = trace_slot(h, DFLASH_KERNEL_FINISH, conv_grid(c, h->n_sm));
    launch_conv(c, h->n_sm, s);
    ck(cudaGetLastError(), "conv finish launch");
  };

  for (int l = 0; l < g.L; ++l) {
    prep_norm(h->at<float>(h->lo.in_ln) + (size_t)l * g.H);
    ck(cudaGetLastError(), "input norm launch");
    if (Gc) conv_prepare(l, 0);

    GemmSpec q;
    q.site = 2 + 4 * l;
    q.W = h->at<char>(h->lo.qkv) + (size_t)l * g.qkv_n * g.H * ew;
    q.wscale = fp8 ? h->at<float>(h->lo.s_qkv) + (size_t)l * g.qkv_n : nullptr;
    q.N = g.qkv_n;
    q.K = g.H;
    q.X = h->at<void>(h->lo.op_h);
    q.xmap = h->xmap_h;
    q.omode = O_RED;
    q.dst = qkv_acc;
    q.dst_ld = g.qkv_n;
    q.e = base_epi(h);
    q.e.n_tok = n_tok;
    run_gemm(h, q, s);

    {
      FinishArgs f = fb;
      f.layer = l;
      f.acc = qkv_acc;
      f.qn = h->at<float>(h->lo.qn) + (size_t)l * g.d;
      f.kn = h->at<float>(h->lo.kn) + (size_t)l * g.d;
      Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * g.qkv_n * 6, s);
      f.trace = trace_slot(h, DFLASH_KERNEL_FINISH, qk_finish_grid(f, h->n_sm));
      launch_qk_finish(f, h->n_sm, s);
    }
    ck(cudaGetLastError(), "qk finish launch");

    // attention over [cached ctx ; block] K/V, split over keys, then merge
    AttnArgs a{};
    a.q = h->at<void>(h->lo.q);
    a.kpool = h->kv->kpool;
    a.vpool = h->kv->vpool;
    a.layer = l;
    a.block_table = h->at<int>(h->lo.btab);
    a.rd = h->at<RoundDesc>(h->lo.rdesc);
    a.part_o = h->at<float>(h->lo.apart_o);
    a.part_ml = h->at<float>(h->lo.apart_ml);
    a.op = h->at<void>(h->lo.op_o);
    a.op_ld = g.Hq * g.d;
    a.op_plane = (long)Mt * g.Hq * g.d;
    a.op_kind = op_kind_of(h->cfg.weight_dtype);
    a.scale_log2 = 1.4426950408889634f / std::sqrt((float)g.d);
    a.err = h->at<int>(h->lo.err);
    a.g = g;
    {
      // warps per merged row from the largest split count (any count merges
      // correctly; this one covers the largest in one pass)
      int max_split = 1;
      for (int i = 0; i < rd.n_seq; ++i) max_split = std::max(max_split, (rd.item0[i + 1] - rd.item0[i]) / g.Hkv);
      a.comb_wpr = attn_combine_wpr(max_split);
      a.comb_max_split = max_split;
    }
    // bytes per cached element (e4m3: the code plus its row's scale share)
    const double ekv = g.kvtype == KV_F32 ? 4 : (g.kvtype == KV_FP8 ? 1.0 + 4.0 / g.d : 2);
    const double part_b = (double)rd.n_items * g.G * kBlock * (g.d + 2) * 4;
    {
      double kv_b = 0;
      for (int i = 0; i < rd.n_seq; ++i) kv_b += (double)(rd.len[i] + kBlock) * g.Hkv * g.d * 2 * ekv;
      Launch L(h, DFLASH_KERNEL_ATTENTION, kv_b + (double)n_tok * g.Hq * g.d * ekv + part_b, s);
      a.trace = h->attn_tc ? trace_slot(h, DFLASH_KERNEL_ATTENTION, rd.n_items) : nullptr;
      if (h->attn_fp8) launch_attention_tc8(a, rd.n_items, &h->qmap, &h->kv->kmap, &h->kv->vmap, s);
      else if (h->attn_tc) launch_attention_tc(a, rd.n_items, &h->qmap, &h->kv->kmap, &h->kv->vmap, s);
      else launch_attention_simt(a, rd.n_items, s);
    }
    ck(cudaGetLastError(), "attention launch");
    {
      Launch L(h, DFLASH_KERNEL_COMBINE, part_b + (double)n_tok * g.Hq * g.d * 4, s);
      a.trace = trace_slot(h, DFLASH_KERNEL_COMBINE, attn_combine_grid(a, n_tok));
      launch_attn_combine(a, n_tok, s);
    }
    ck(cudaGetLastError(), "attention combine launch");

    GemmSpec o;
    o.site = 3 + 4 * l;
    o.W = h->at<char>(h->lo.o) + (size_t)l * g.H * g.Hq * g.d * ew;
    o.wscale = fp8 ? h->at<float>(h->lo.s_o) + (size_t)l * g.H : nullptr;
    o.N = g.H;
    o.K = g.Hq * g.d;
    o.X = h->at<void>(h->lo.op_o);
    o.xmap = h->xmap_o;
    o.omode = O_RED;
    o.dst = Gc ? cy : hres;
    o.dst_ld = g.H;
    o.e = base_epi(h);
    o.e.n_tok = n_tok;
    run_gemm(h, o, s);
    if (Gc) conv_finish(l, 0);

    if (fused_mlp) {
      // post-attention RMSNorm, gate/up and SwiGLU in one tile-owning launch
      OwnArgs oa{};
      oa.W = h->at<uint8_t>(h->lo.gu) + (size_t)l * 2 * g.I * g.H * ew;
      oa.n_tiles = 2 * g.I / kTileN;
      oa.kb = g.H / kTileK;
      oa.n_tok = n_tok;
      oa.gain = h->at<float>(h->lo.post_ln) + (size_t)l * g.H;
      oa.wscale = fp8 ? h->at<float>(h->lo.s_gu) + (size_t)l * 2 * g.I : nullptr;
      oa.epi = OWN_SWIGLU;
      oa.out = h->at<void>(h->lo.op_a);
      oa.out_ld = g.I;
      oa.out_plane = (long)Mt * g.I;
      oa.err = h->at<int>(h->lo.err);
      oa.g = g;
      const double bytes = (double)2 * g.I * g.H * ew + (fp8 ? 2.0 * g.I * 4 : 0.0) +
                           (double)oa.n_tiles * n_tok * g.H * 4 + (double)n_tok * g.I * 4;
      Launch L(h, DFLASH_KERNEL_GEMM, bytes, s);
      oa.trace = trace_slot(h, DFLASH_KERNEL_GEMM, oa.n_tiles);
      ck(launch_proj_own(oa, &h->hmap[n_tok > 16 ? 1 : 0], s), "fused gate/up launch");
    } else {
    prep_norm(h->at<float>(h->lo.post_ln) + (size_t)l * g.H);
    ck(cudaGetLastError(), "post norm launch");
    if (Gc) conv_prepare(l, 1);

    GemmSpec gu;
    gu.site = 4 + 4 * l;
    gu.W = h->at<char>(h->lo.gu) + (size_t)l * 2 * g.I * g.H * ew;
    gu.wscale = fp8 ? h->at<float>(h->lo.s_gu) + (size_t)l * 2 * g.I : nullptr;
    gu.N = 2 * g.I;
    gu.K = g.H;
    gu.X = h->at<void>(h->lo.op_h);
    gu.xmap = h->xmap_h;
    gu.omode = O_RED;
    gu.dst = gu_acc;
    gu.dst_ld = 2 * g.I;
    gu.e = base_epi(h);
    gu.e.n_tok = n_tok;
    run_gemm(h, gu, s);

    {
      FinishArgs f = fb;
      f.acc = gu_acc;
      f.op = h->at<void>(h->lo.op_a);
      f.op_plane = (long)Mt * g.I;
      Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * g.I * 16, s);
      f.trace = trace_slot(h, DFLASH_KERNEL_FINISH, swiglu_grid(f, h->n_sm));
      launch_swiglu(f, h->n_sm, s);
    }
    ck(cudaGetLastError(), "swiglu launch");
    }

    GemmSpec dn;
    dn.site = 5 + 4 * l;
    dn.W = h->at<char>(h->lo.down) + (size_t)l * g.H * g.I * ew;
    dn.wscale = fp8 ? h->at<float>(h->lo.s_down) + (size_t)l * g.H : nullptr;
    dn.N = g.H;
    dn.K = g.I;
    dn.X = h->at<void>(h->lo.op_a);
    dn.xmap = h->xmap_a;
    dn.omode = O_RED;
    dn.dst = Gc ? cy : hres;
    dn.dst_ld = g.H;
    dn.e = base_epi(h);
    dn.e.n_tok = n_tok;
    run_gemm(h, dn, s);
    if (Gc) conv_finish(l, 1);
  }
  {
    Launch L(h, DFLASH_KERNEL_NORM, (double)n_tok * g.H * 8, s);
    launch_final_norm(hres, h->at<float>(h->lo.fn), out, n_tok, g, trace_slot(h, DFLASH_KERNEL_NORM, n_tok), s);
  }
  ck(cudaGetLastError(), "final norm launch");
}

// Fill the attention split plan of a round descriptor.
void plan_attention(dflash_t* h, RoundDesc& rd, const std::vector<int64_t>& lens) {
  const AttnPlanCtx c = attn_plan_ctx(h->g.Hkv, h->lo.items_cap, h->n_sm, h->attn_tc, rd.n_seq * kBlock);
  rd.split_pages = plan_items(c, attended_pages(lens, rd.kstart), rd.item0, rd.perm);
  rd.n_items = rd.item0[rd.n_seq];   // more than items_cap: refused by the caller
}


template <class F>
int guarded(F&& f) {
  try {
    return f();
  } catch (const CudaError& e) {
    return fail(DFLASH_ERR_CUDA, "%s", e.what.c_str());
  } catch (const std::bad_alloc&) {
    return fail(DFLASH_ERR_CAPACITY, "host allocation failed");
  }
}

int check_seq_ids(dflash_t* h, int n_seq, const int32_t* ids) {
  std::vector<char> seen(h->cfg.max_seqs, 0);
  for (int i = 0; i < n_seq; ++i) {
    if (ids[i] < 0 || ids[i] >= h->cfg.max_seqs) return fail(DFLASH_ERR_INVALID_ARG, "seq id %d out of range", ids[i]);
    if (seen[ids[i]]) return fail(DFLASH_ERR_INVALID_ARG, "seq id %d repeated", ids[i]);
    seen[ids[i]] = 1;
  }
  return DFLASH_OK;
}

// Context window: keep the most recent ctx_cap positions of a sequence.
// Pages wholly before the window return to the pool; keys before the window
// in its first page are masked by the attention.  The first-light forward's
// internal slot keeps its whole context.
void evict_window(dflash_t* h, int slot) {
  if (h->ctx_cap <= 0 || slot >= h->cfg.max_seqs) return;
  const int64_t ks = std::max<int64_t>(h->kstart[slot], h->len[slot] - h->ctx_cap);
  if (ks <= h->kstart[slot]) return;
  h->kstart[slot] = ks;
  auto& pl = h->pages[slot];
  for (int64_t i = 0; i < ks / kPage && i < (int64_t)pl.size(); ++i)
    if (pl[i] >= 0) {
      h->kv->free_pages.push_back(pl[i]);
      pl[i] = -1;
    }
  h->evicted_any = true;
}

// Validated ingest of rows into explicit slots (used by the public entry and
// by forward_full's internal slot).
int ingest_slots(dflash_t* h, int n_seq, const int32_t* slots, const int32_t* t_per_seq, const int32_t* pos_new,
                 const float* taps, cudaStream_t s) {
  long total = 0;
  for (int i = 0; i < n_seq; ++i) {
    if (t_per_seq[i] < 0) return fail(DFLASH_ERR_INVALID_ARG, "negative row count");
    total += t_per_seq[i];
  }
  if (total == 0) return DFLASH_OK;
  if (total > h->cfg.max_ingest_rows)
    return fail(DFLASH_ERR_CAPACITY, "ingest of %ld rows exceeds max_ingest_rows %d", total, h->cfg.max_ingest_rows);
  if (!taps || !pos_new) return fail(DFLASH_ERR_INVALID_ARG, "taps / pos_new is null");
  if (!aligned16(taps)) return fail(DFLASH_ERR_INVALID_ARG, "taps must start on a 16-byte boundary");
  for (int i = 0; i < n_seq; ++i)
    if (h->len[slots[i]] + t_per_seq[i] + kBlock > h->cfg.max_seq_len)
      return fail(DFLASH_ERR_CAPACITY, "sequence %d would exceed max_seq_len %d", slots[i], h->cfg.max_seq_len);
  InitBlob* blob = new InitBlob();
  std::vector<int> taken;
  blob->n_pt = 0;
  IngestDesc& id = blob->ingest;
  id.n_rows = (int)total;
  int r = 0;
  for (int i = 0; i < n_seq; ++i) {
    const int slot = slots[i];
    if (!ensure_pages(h, slot, h->len[slot] + t_per_seq[i], *blob, taken)) {
      rollback_pages(h, *blob, taken);
      delete blob;
      return fail(DFLASH_ERR_CAPACITY, "out of KV pages");
    }
    for (int j = 0; j < t_per_seq[i]; ++j, ++r) {
      const int64_t row = h->len[slot] + j;
      id.row_dest[r] = h->pages[slot][row / kPage] * kPage + (int)(row % kPage);
      id.row_pos[r] = pos_new[r];
    }
  }
  int rc = guarded([&]() -> int {
    enqueue_ingest(h, *blob, taps, s);
    return DFLASH_OK;
  });
  if (rc != DFLASH_OK) {
    rollback_pages(h, *blob, taken);
    delete blob;
    return rc;
  }
  for (int i = 0; i < n_seq; ++i) {
    h->len[slots[i]] += t_per_seq[i];
    evict_window(h, slots[i]);
  }
  h->last_stream = s;
  delete blob;
  return DFLASH_OK;
}

// A round through a cached graph: the ~80 launches of the per-step path cost
// the host about as long as the GPU takes to run them, so they are captured
// once per (sequences, attention items, KV region) and replayed; a replay
// changes only the init node (descriptor blob, noise rows) and the final-norm
// node (output rows).  Off while profiling and when the caller's stream is
// itself being captured; while tracing, each round is captured afresh with
// its own trace regions.
void enqueue_round_graph(dflash_t* h, InitBlob& blob, const float* noise, float* out, cudaStream_t s) {
  const RoundDesc& rd = blob.round;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  ck(cudaStreamIsCapturing(s, &cap), "stream capture query");
  if (h->prof_on || cap != cudaStreamCaptureStatusNone) {
    enqueue_round(h, blob, noise, out, s);
    return;
  }
  if (h->trace_buf) {
    // a traced round runs the same graph as an untraced one, captured afresh
    // with this round's trace regions and discarded after its launch
    if (!h->cap_stream) ck(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking), "capture stream");
    ck(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeRelaxed), "traced round capture begin");
    cudaGraph_t tg = nullptr;
    try {
      enqueue_round(h, blob, noise, out, h->cap_stream);
    } catch (...) {
      cudaStreamEndCapture(h->cap_stream, &tg);
      if (tg) cudaGraphDestroy(tg);
      throw;
    }
    ck(cudaStreamEndCapture(h->cap_stream, &tg), "traced round capture end");
    cudaGraphExec_t te = nullptr;
    cudaError_t ie = cudaGraphInstantiate(&te, tg, 0);
    cudaGraphDestroy(tg);
    ck(ie, "traced round instantiate");
    h->traced_execs.push_back(te);   // released when tracing stops (after a device sync)
    ck(cudaGraphLaunch(te, s), "traced round launch");
    return;
  }
  const void* region = h->kv;
  dflash_handle::RoundGraph* gr = nullptr;
  for (auto& e : h->graphs)
    if (e.n_seq == rd.n_seq && e.n_items == rd.n_items && e.region == region) gr = &e;
  InitArgs ia = round_init_args(h, rd, noise);
  if (gr) {
    cudaKernelNodeParams p = gr->init_p;
    void* ip[2] = {&ia, &blob};
    p.kernelParams = ip;
    ck(cudaGraphExecKernelNodeSetParams(gr->exec, gr->init_node, &p), "round graph init update");
    const float* hres = h->at<float>(h->lo.h);
    const float* fn = h->at<float>(h->lo.fn);
    int H = h->g.H;
    float eps = h->g.eps;
    unsigned long long* no_trace = nullptr;
    cudaKernelNodeParams q = gr->norm_p;
    void* np[6] = {&hres, &fn, &out, &H, &eps, &no_trace};
    q.kernelParams = np;
    ck(cudaGraphExecKernelNodeSetParams(gr->exec, gr->norm_node, &q), "round graph output update");
    ck(cudaGraphLaunch(gr->exec, s), "round graph launch");
    h->launches += gr->launches;
    gr->used = ++h->graph_clock;
    return;
  }
  // capture this round on the private stream (the caller's may be the legacy
  // default stream, which cannot be captured), keep it, and run it on the
  // caller's stream
  if (!h->cap_stream) ck(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking), "capture stream");
  cudaStream_t cs = h->cap_stream;
  const int64_t l0 = h->launches;
  ck(cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed), "round capture begin");
  cudaGraph_t graph = nullptr;
  try {
    enqueue_round(h, blob, noise, out, cs);
  } catch (...) {
    cudaStreamEndCapture(cs, &graph);
    if (graph) cudaGraphDestroy(graph);
    throw;
  }
  ck(cudaStreamEndCapture(cs, &graph), "round capture end");
  dflash_handle::RoundGraph e;
  e.n_seq = rd.n_seq;
  e.n_items = rd.n_items;
  e.region = region;
  e.launches = h->launches - l0;
  size_t n = 0;
  ck(cudaGraphGetNodes(graph, nullptr, &n), "round graph nodes");
  std::vector<cudaGraphNode_t> nodes(n);
  ck(cudaGraphGetNodes(graph, nodes.data(), &n), "round graph nodes");
  for (auto nd : nodes) {
    cudaGraphNodeType t;
    ck(cudaGraphNodeGetType(nd, &t), "round graph node type");
    if (t != cudaGraphNodeTypeKernel) continue;
    cudaKernelNodeParams p{};
    ck(cudaGraphKernelNodeGetParams(nd, &p), "round graph node params");
    if (p.func == init_kernel_entry()) {
      e.init_node = nd;
      e.init_p = p;
    } else if (p.func == final_norm_kernel_entry()) {
      e.norm_node = nd;
      e.norm_p = p;
    }
  }
  if (!e.init_node || !e.norm_node) {
    cudaGraphDestroy(graph);
    throw CudaError{"round graph: init or final-norm node not found"};
  }
  cudaError_t ie = cudaGraphInstantiate(&e.exec, graph, 0);
  if (ie != cudaSuccess) {
    cudaGraphDestroy(graph);
    throw CudaError{std::string("round graph instantiate: ") + cudaGetErrorString(ie)};
  }
  // node handles of the source graph address the same nodes in the exec graph
  // for parameter updates, so the source graph stays alive with it
  e.used = ++h->graph_clock;
  if (h->graphs.size() >= 8) {   // drop the least recently used
    auto it = std::min_element(h->graphs.begin(), h->graphs.end(),
                               [](const dflash_handle::RoundGraph& a, const dflash_handle::RoundGraph& b) {
                                 return a.used < b.used;
                               });
    cudaGraphExecDestroy(it->exec);
    cudaGraphDestroy(it->graph);
    h->graphs.erase(it);
  }
  e.graph = graph;
  h->graphs.push_back(e);
  ck(cudaGraphLaunch(e.exec, s), "round graph launch");
}

int round_slots(dflash_t* h, int n_seq, const int32_t* slots, const int32_t* pos_block, const float* noise,
                float* out, cudaStream_t s) {
  if (!pos_block || !noise || !out) return fail(DFLASH_ERR_INVALID_ARG, "pos_block / noise_emb / out is null");
  if (!aligned16(noise) || !aligned16(out))
    return fail(DFLASH_ERR_INVALID_ARG, "noise_emb / out must start on a 16-byte boundary");
  InitBlob* blob = new InitBlob();
  std::vector<int> taken;
  blob->n_pt = 0;
  RoundDesc& rd = blob->round;
  rd.n_seq = n_seq;
  rd.n_tok = n_seq * kBlock;
  std::vector<int64_t> lens(n_seq);
  for (int i = 0; i < n_seq; ++i) {
    const int slot = slots[i];
    lens[i] = h->len[slot];
    rd.seq_slot[i] = slot;
    rd.len[i] = (int)lens[i];
    rd.kstart[i] = (int)h->kstart[slot];
    for (int j = 0; j < kBlock; ++j) rd.pos[i * kBlock + j] = pos_block[i * kBlock + j];
    if (!ensure_pages(h, slot, lens[i] + kBlock, *blob, taken)) {
      rollback_pages(h, *blob, taken);
      delete blob;
      return fail(DFLASH_ERR_CAPACITY, "out of KV pages for the block rows");
    }
    for (int j = 0; j < kBlock; ++j) {
      const int64_t row = lens[i] + j;
      rd.dest[i * kBlock + j] = h->pages[slot][row / kPage] * kPage + (int)(row % kPage);
    }
  }
  plan_attention(h, rd, lens);
  if (rd.n_items > h->lo.items_cap) {
    rollback_pages(h, *blob, taken);
    delete blob;
    return fail(DFLASH_ERR_CAPACITY, "attention plan exceeds its scratch");
  }
  int rc = guarded([&]() -> int {
    enqueue_round_graph(h, *blob, noise, out, s);
    return DFLASH_OK;
  });
  if (rc != DFLASH_OK) rollback_pages(h, *blob, taken);
  else h->last_stream = s;
  delete blob;
  return rc;
}

void release_slot(dflash_t* h, int slot) {
  for (int p : h->pages[slot])
    if (p >= 0) h->kv->free_pages.push_back(p);
  h->pages[slot].clear();
  h->len[slot] = 0;
  h->kstart[slot] = 0;
}

// Makes `r` the region the enqueued kernels use (pools, maps, free list and
// the device geometry's pages-per-layer) until the scope ends.
// e4m3 pools: K pages [64 keys][d bytes] in the 128-byte swizzle (the score
// MMA's B operand as stored), V^T pages [d][64 bytes] unswizzled (threads
// convert them to f16); the maps cover the codes, not the scales after them.
void kv_maps_fp8(dflash_handle::KvRegion& r, const void* kpool, const void* vpool, uint64_t rows, int d) {
  r.kmap = make_map_u8(kpool, rows * kPage, (uint64_t)d, kPage, (uint32_t)d, CU_TENSOR_MAP_SWIZZLE_128B);
  r.vmap = make_map_u8(vpool, rows * d, kPage, (uint32_t)d, kPage, CU_TENSOR_MAP_SWIZZLE_NONE);
}

struct RegionScope {
  dflash_t* h;
  dflash_handle::KvRegion* prev;
  int prev_pages;
  RegionScope(dflash_t* h_, dflash_handle::KvRegion* r) : h(h_), prev(h_->kv), prev_pages(h_->g.max_pages) {
    h->kv = r;
    h->g.max_pages = r->max_pages;
  }
  ~RegionScope() {
    h->kv = prev;
    h->g.max_pages = prev_pages;
  }
};

// Ingest ctx rows into the internal slot in max_ingest_rows chunks, run the
// block forward, release the slot (the body of both first-light entries).
int first_light(dflash_t* h, int32_t ctx, const float* taps, const float* noise_emb, const int32_t* pos,
                float* out, cudaStream_t s) {
  const int slot = h->cfg.max_seqs;
  int rc = DFLASH_OK;
  const int chunk = h->cfg.max_ingest_rows;
  const size_t width = (size_t)h->g.n * h->g.H;
  for (int r0 = 0; r0 < ctx && rc == DFLASH_OK; r0 += chunk) {
    const int t = std::min(chunk, ctx - r0);
    rc = ingest_slots(h, 1, &slot, &t, pos + r0, taps + (size_t)r0 * width, s);
  }
  if (rc == DFLASH_OK) rc = round_slots(h, 1, &slot, pos + ctx, noise_emb, out, s);
  release_slot(h, slot);
  return rc;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* dflash_last_error(void) { return g_last_error.c_str(); }

int dflash_workspace_bytes(const dflash_config* cfg, size_t* bytes) {
  g_last_error.clear();
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (!bytes) return fail(DFLASH_ERR_INVALID_ARG, "bytes is null");
  *bytes = make_layout(*cfg, sm_count()).total;
  return DFLASH_OK;
}

int dflash_attention_plan(const dflash_config* cfg, int32_t n_sm, int32_t n_seq, const int64_t* lens,
                          const int64_t* kstart, int32_t* split_pages, int32_t* n_items, int32_t* item0,
                          int32_t* launch_order, int32_t max_items) {
  g_last_error.clear();
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (n_sm < 0) return fail(DFLASH_ERR_INVALID_ARG, "n_sm must be >= 0");
  if (n_seq < 1 || n_seq > cfg->max_batch) return fail(DFLASH_ERR_INVALID_ARG, "n_seq must be 1..max_batch");
  if (!lens || !split_pages || !n_items) return fail(DFLASH_ERR_INVALID_ARG, "lens, split_pages and n_items are required");
  if (launch_order && max_items < 0) return fail(DFLASH_ERR_INVALID_ARG, "max_items must be >= 0");
  if (n_sm == 0) n_sm = sm_count();
  std::vector<int64_t> L(lens, lens + n_seq);
  std::vector<int> ks(n_seq, 0);
  for (int i = 0; i < n_seq; ++i) {
    if (L[i] < 0 || L[i] + kBlock > cfg->max_seq_len)
      return fail(DFLASH_ERR_INVALID_ARG, "lens[%d] must be 0..max_seq_len - 16", i);
    const int64_t k = kstart ? kstart[i] : 0;
    if (k < 0 || k > L[i]) return fail(DFLASH_ERR_INVALID_ARG, "kstart[%d] must be 0..lens[%d]", i, i);
    ks[i] = (int)k;
  }
  const AttnPlanCtx c = attn_plan_ctx(cfg->n_kv_heads, items_capacity(*cfg, n_sm), n_sm,
                                      cfg->kv_dtype != DFLASH_F32, n_seq * kBlock);
  std::vector<int> i0(n_seq + 1);
  std::vector<uint16_t> order(kMaxItems);
  *split_pages = plan_items(c, attended_pages(L, ks.data()), i0.data(), order.data());
  *n_items = i0[n_seq];
  if (item0) std::copy(i0.begin(), i0.end(), item0);
  if (*n_items > c.items_cap)
    return fail(DFLASH_ERR_CAPACITY, "the plan's %d items exceed the scratch's %ld", *n_items, c.items_cap);
  if (launch_order) {
    if (max_items < *n_items) return fail(DFLASH_ERR_CAPACITY, "launch_order holds %d of %d items", max_items, *n_items);
    std::copy(order.begin(), order.begin() + *n_items, launch_order);
  }
  return DFLASH_OK;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, void* workspace, size_t ws_bytes, void* stream,
                  dflash_t** out) {
  g_last_error.clear();
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (!w || !workspace || !out) return fail(DFLASH_ERR_INVALID_ARG, "weights / workspace / out is null");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DFLASH_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const bool fp8 = cfg->weight_dtype == DFLASH_FP8_E4M3;
  if (!w->fc || !w->hidden_norm || !w->norm || !w->layers || (fp8 && !w->fc_scale))
    return fail(DFLASH_ERR_INVALID_ARG, "missing top-level weight tensor");
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    if (!L.q || !L.k || !L.v || !L.o || !L.gate || !L.up || !L.down || !L.q_norm || !L.k_norm || !L.input_ln ||
        !L.post_ln)
      return fail(DFLASH_ERR_INVALID_ARG, "missing tensor in layer %d", l);
    if (fp8 && (!L.q_scale || !L.k_scale || !L.v_scale || !L.o_scale || !L.gate_scale || !L.up_scale || !L.down_scale))
      return fail(DFLASH_ERR_INVALID_ARG, "missing fp8 scale in layer %d", l);
    if (cfg->conv_groups > 0)
      for (int sub = 0; sub < 2; ++sub) {
        if (!L.conv_base[sub] || !L.conv_dyn[sub] || (fp8 && !L.conv_dyn_scale[sub]))
          return fail(DFLASH_ERR_INVALID_ARG, "missing DFlash2 conv tensor in layer %d", l);
        if (cfg->weight_dtype != DFLASH_F32 && !aligned16(L.conv_dyn[sub]))
          return fail(DFLASH_ERR_INVALID_ARG, "conv_dyn must start on a 16-byte boundary");
      }
    // bf16 and e4m3 matrices are re-blocked with 16- and 8-byte moves
    if (cfg->weight_dtype != DFLASH_F32 &&
        !(aligned16(L.q) && aligned16(L.k) && aligned16(L.v) && aligned16(L.o) && aligned16(L.gate) &&
          aligned16(L.up) && aligned16(L.down)))
      return fail(DFLASH_ERR_INVALID_ARG, "bf16 weight matrices must start on a 16-byte boundary (layer %d)", l);
  }
  if (cfg->weight_dtype != DFLASH_F32 && !aligned16(w->fc))
    return fail(DFLASH_ERR_INVALID_ARG, "bf16 weight matrices must start on a 16-byte boundary (fc)");
  const int n_sm = sm_count();
  Layout lo = make_layout(*cfg, n_sm);
  if (ws_bytes < lo.total) return fail(DFLASH_ERR_CAPACITY, "workspace %zu bytes < required %zu", ws_bytes, lo.total);

  dflash_t* h = new (std::nothrow) dflash_handle();
  if (!h) return fail(DFLASH_ERR_CAPACITY, "host allocation failed");
  h->cfg = *cfg;
  {
    static std::atomic<uint64_t> next_uid{1};
    h->uid = next_uid.fetch_add(1);
  }
  h->lo = lo;
  h->ws = static_cast<char*>(workspace);
  h->n_sm = n_sm;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    delete h;
    return fail(DFLASH_ERR_CUDA, "device query failed");
  }
  const int L = cfg->n_layers, H = cfg->hidden, d = cfg->head_dim, Hq = cfg->n_heads, Hkv = cfg->n_kv_heads;
  const int I = cfg->intermediate;
  Geo& g = h->g;
  g.L = L; g.H = H; g.Hq = Hq; g.Hkv = Hkv; g.d = d; g.I = I; g.n = cfg->n_taps; g.G = Hq / Hkv;
  g.qkv_n = (Hq + 2 * Hkv) * d;
  g.kv_n = 2 * Hkv * d;
  g.Mt = lo.Mt;
  g.wtype = cfg->weight_dtype;
  g.kvtype = cfg->kv_dtype;
  g.max_pages = cfg->max_pages;
  g.pages_per_seq = lo.pps;
  g.eps = (float)cfg->rms_eps;
  std::vector<double> inv;
  rope_table(*cfg, inv, g.mscale);
  h->len.assign(cfg->max_seqs + 1, 0);
  h->pages.assign(cfg->max_seqs + 1, {});
  h->kstart.assign(cfg->max_seqs + 1, 0);
  h->pool.kpool = h->ws + lo.kpool;
  h->pool.vpool = h->ws + lo.vpool;
  h->pool.max_pages = cfg->max_pages;
  h->pool.free_pages.resize(cfg->max_pages);
  for (int i = 0; i < cfg->max_pages; ++i) h->pool.free_pages[i] = cfg->max_pages - 1 - i;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = guarded([&]() -> int {
    const size_t ew = esize_w(cfg->weight_dtype);
    auto cp = [&](size_t dst_off, const void* src, size_t bytes) {
      ck(cudaMemcpyAsync(h->ws + dst_off, src, bytes, cudaMemcpyDeviceToDevice, s), "weight copy");
    };
    // A matrix piece: source rows i land on logical rows base + (i / chunk) *
    // stride + i % chunk of the [N][K] matrix at dst_off (row-major, or in
    // 16 KB swizzled blocks for the tensor-core path).
    const bool tc = cfg->weight_dtype != DFLASH_F32;
    auto mat = [&](size_t dst_off, int K, const void* src, int n_rows, int chunk, int stride, int base) {
      if (tc) {
        if (fp8) launch_repack_e4m3(h->ws + dst_off, K, src, n_rows, chunk, stride, base, s);
        else launch_repack(h->ws + dst_off, K, src, n_rows, chunk, stride, base, s);
        ck(cudaGetLastError(), "weight repack");
      } else if (chunk == n_rows) {
        cp(dst_off + (size_t)base * K * ew, src, (size_t)n_rows * K * ew);
      } else {
        const size_t cb = (size_t)chunk * K * ew;
        ck(cudaMemcpy2DAsync(h->ws + dst_off + (size_t)base * K * ew, (size_t)stride * K * ew, src, cb, cb,
                             n_rows / chunk, cudaMemcpyDeviceToDevice, s),
           "interleaved weight copy");
      }
    };
    if (cfg->conv_groups > 0) {
      // padding rows of the dynamic projections stay zero
      ck(cudaMemsetAsync(h->ws + lo.cdyn, 0, lo.s_cdyn - lo.cdyn, s), "conv projection clear");
      if (fp8) ck(cudaMemsetAsync(h->ws + lo.s_cdyn, 0, lo.cu - lo.s_cdyn, s), "conv scale clear");
    }
    mat(lo.fc, g.n * H, w->fc, H, H, 0, 0);
    if (fp8) cp(lo.s_fc, w->fc_scale, (size_t)H * 4);
    cp(lo.hn, w->hidden_norm, (size_t)H * 4);
    cp(lo.fn, w->norm, (size_t)H * 4);
    for (int l = 0; l < L; ++l) {
      const dflash_layer_weights& W = w->layers[l];
      const int qr = Hq * d, kr = Hkv * d;
      const size_t qkv0 = lo.qkv + (size_t)l * g.qkv_n * H * ew;
      mat(qkv0, H, W.q, qr, qr, 0, 0);
      mat(qkv0, H, W.k, kr, kr, 0, qr);
      mat(qkv0, H, W.v, kr, kr, 0, qr + kr);
      mat(lo.kvall, H, W.k, kr, kr, 0, l * g.kv_n);
      mat(lo.kvall, H, W.v, kr, kr, 0, l * g.kv_n + kr);
      mat(lo.o + (size_t)l * H * Hq * d * ew, Hq * d, W.o, H, H, 0, 0);
      if (cfg->conv_groups > 0) {
        const int nd = 4 * cfg->conv_groups;
        for (int sub = 0; sub < 2; ++sub) {
          const size_t m = (size_t)l * 2 + sub;
          cp(lo.cbase + m * 2 * H * 2 * 4, W.conv_base[sub], (size_t)2 * H * 2 * 4);
          mat(lo.cdyn + m * lo.conv_n * H * ew, H, W.conv_dyn[sub], nd, nd, 0, 0);
          if (fp8) cp(lo.s_cdyn + m * lo.conv_n * 4, W.conv_dyn_scale[sub], (size_t)nd * 4);
        }
      }
      mat(lo.down + (size_t)l * H * I * ew, I, W.down, H, H, 0, 0);
      // gate/up interleaved in blocks of 64 rows: [g0..63, u0..63, g64..127, u64..127, ...]
      const size_t gu0 = lo.gu + (size_t)l * 2 * I * H * ew;
      mat(gu0, H, W.gate, I, 64, 128, 0);
      mat(gu0, H, W.up, I, 64, 128, 64);
      cp(lo.in_ln + (size_t)l * H * 4, W.input_ln, (size_t)H * 4);
      cp(lo.post_ln + (size_t)l * H * 4, W.post_ln, (size_t)H * 4);
      cp(lo.qn + (size_t)l * d * 4, W.q_norm, (size_t)d * 4);
      cp(lo.kn + (size_t)l * d * 4, W.k_norm, (size_t)d * 4);
      if (fp8) {
        const size_t sq0 = lo.s_qkv + (size_t)l * g.qkv_n * 4;
        cp(sq0, W.q_scale, qr * 4);
        cp(sq0 + qr * 4, W.k_scale, kr * 4);
        cp(sq0 + (qr + kr) * 4, W.v_scale, kr * 4);
        const size_t sk0 = lo.s_kvall + (size_t)l * g.kv_n * 4;
        cp(sk0, W.k_scale, kr * 4);
        cp(sk0 + kr * 4, W.v_scale, kr * 4);
        cp(lo.s_o + (size_t)l * H * 4, W.o_scale, (size_t)H * 4);
        cp(lo.s_down + (size_t)l * H * 4, W.down_scale, (size_t)H * 4);
        const size_t sb = 64 * 4, sgu0 = lo.s_gu + (size_t)l * 2 * I * 4;
        ck(cudaMemcpy2DAsync(h->ws + sgu0, 2 * sb, W.gate_scale, sb, sb, I / 64, cudaMemcpyDeviceToDevice, s), "gate scale");
        ck(cudaMemcpy2DAsync(h->ws + sgu0 + sb, 2 * sb, W.up_scale, sb, sb, I / 64, cudaMemcpyDeviceToDevice, s), "up scale");
      }
    }
    ck(cudaMemcpyAsync(h->ws + lo.inv_freq, inv.data(), inv.size() * 8, cudaMemcpyHostToDevice, s), "rope table");
    h->use_tc = cfg->weight_dtype != DFLASH_F32;
    h->attn_tc = cfg->kv_dtype != DFLASH_F32;
    h->attn_fp8 = cfg->kv_dtype == DFLASH_FP8_E4M3;
    if (h->use_tc) {
      const uint64_t Mt2 = 2ull * lo.Mt;
      const uint32_t tall = Mt2 >= 256 ? 128u : 16u;   // 128-row boxes only where a pass can reach 128 tokens
      for (int b = 0; b < 2; ++b) {
        const uint32_t box = b ? tall : 16u;
        h->xmap_taps[b] = make_map_bf16(h->ws + lo.op_taps, Mt2, (uint64_t)g.n * H, box);
        h->xmap_h[b] = make_map_bf16(h->ws + lo.op_h, Mt2, H, box);
        h->xmap_o[b] = make_map_bf16(h->ws + lo.op_o, Mt2, (uint64_t)Hq * d, box);
        h->xmap_a[b] = make_map_bf16(h->ws + lo.op_a, Mt2, I, box);
      }
      for (int b = 0; b < 2; ++b) h->hmap[b] = make_map_f32(h->ws + lo.h, (uint64_t)lo.Mt, H, b ? 32u : 16u);
    }
    if (h->attn_tc) {
      const uint64_t pool_rows = (uint64_t)L * cfg->max_pages * Hkv;
      // queries: bf16 beside a bf16 cache, f16 beside an e4m3 one (2-byte
      // elements either way; the copy does not convert)
      h->qmap = make_map_bf16_3d(h->ws + lo.q, d, Hq, lo.Mt, Hq / Hkv, kBlock);
      if (h->attn_fp8) {
        kv_maps_fp8(h->pool, h->ws + lo.kpool, h->ws + lo.vpool, pool_rows, d);
      } else {
        h->pool.kmap = make_map_bf16(h->ws + lo.kpool, pool_rows * kPage, d, kPage);
        h->pool.vmap = make_map_bf16(h->ws + lo.vpool, pool_rows * d, kPage, d);
      }
    }
    // stale pool rows are read (and masked) by the attention MMA: keep them finite
    ck(cudaMemsetAsync(h->ws + lo.kpool, 0, lo.vpool - lo.kpool, s), "K pool clear");
    ck(cudaMemsetAsync(h->ws + lo.vpool, 0, lo.btab - lo.vpool, s), "V pool clear");
    ck(cudaMemsetAsync(h->ws + lo.btab, 0xff, (size_t)(cfg->max_seqs + 1) * lo.pps * 4, s), "block table");
    ck(cudaMemsetAsync(h->ws + lo.counters, 0, (size_t)lo.n_sites * lo.max_tiles * 4, s), "counters");
    ck(cudaMemsetAsync(h->ws + lo.gacc, 0, (size_t)lo.max_tiles * kTileN * kPassTok * 4, s), "tile accumulators");
    ck(cudaMemsetAsync(h->ws + lo.qkv_acc, 0, (size_t)lo.Mt * g.qkv_n * 4, s), "QKV accumulator");
    ck(cudaMemsetAsync(h->ws + lo.gu_acc, 0, (size_t)lo.Mt * 2 * I * 4, s), "gate/up accumulator");
    ck(cudaMemsetAsync(h->ws + lo.err, 0, 256, s), "error word");
    if (cfg->conv_groups > 0)
      ck(cudaMemsetAsync(h->ws + lo.cu, 0, lo.rdesc - lo.cu, s), "conv rows and coefficients");
    ck(cudaStreamSynchronize(s), "create sync");
    return DFLASH_OK;
  });
  if (rc != DFLASH_OK) {
    delete h;
    return rc;
  }
  h->last_stream = s;
  *out = h;
  return DFLASH_OK;
}

int dflash_ingest_ctx(dflash_t* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* t_per_seq,
                      const int32_t* pos_new, const float* taps, void* stream) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (n_seq < 0 || n_seq > h->cfg.max_seqs) return fail(DFLASH_ERR_INVALID_ARG, "n_seq %d out of range", n_seq);
  if (n_seq == 0) return DFLASH_OK;
  if (!seq_ids || !t_per_seq) return fail(DFLASH_ERR_INVALID_ARG, "seq_ids / t_per_seq is null");
  int rc = check_seq_ids(h, n_seq, seq_ids);
  if (rc) return rc;
  return ingest_slots(h, n_seq, seq_ids, t_per_seq, pos_new, taps, static_cast<cudaStream_t>(stream));
}

int dflash_forward_round(dflash_t* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* pos_block,
                         const float* noise_emb, float* out, void* stream) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (n_seq < 1 || n_seq > h->cfg.max_batch)
    return fail(DFLASH_ERR_INVALID_ARG, "n_seq %d not in 1..max_batch (%d)", n_seq, h->cfg.max_batch);
  if (!seq_ids) return fail(DFLASH_ERR_INVALID_ARG, "seq_ids is null");
  int rc = check_seq_ids(h, n_seq, seq_ids);
  if (rc) return rc;
  return round_slots(h, n_seq, seq_ids, pos_block, noise_emb, out, static_cast<cudaStream_t>(stream));
}

int dflash_forward_full(dflash_t* h, int32_t ctx, const float* taps, const float* noise_emb, const int32_t* pos,
                        float* out, void* stream) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (ctx < 0) return fail(DFLASH_ERR_INVALID_ARG, "negative ctx");
  if (!pos || !noise_emb || !out || (ctx > 0 && !taps)) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (!aligned16(noise_emb) || !aligned16(out) || (ctx > 0 && !aligned16(taps)))
    return fail(DFLASH_ERR_INVALID_ARG, "taps / noise_emb / out must start on a 16-byte boundary");
  if (ctx + kBlock > h->cfg.max_seq_len) return fail(DFLASH_ERR_CAPACITY, "ctx exceeds max_seq_len");
  const int need = (ctx + kBlock + kPage - 1) / kPage;
  if ((int)h->kv->free_pages.size() < need) return fail(DFLASH_ERR_CAPACITY, "out of KV pages");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  release_slot(h, h->cfg.max_seqs);
  return first_light(h, ctx, taps, noise_emb, pos, out, s);
}

int dflash_forward_full_static(dflash_t* h, int32_t ctx, const float* taps, const float* noise_emb,
                               const int32_t* pos, float* out, void* stream) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (ctx < 0) return fail(DFLASH_ERR_INVALID_ARG, "negative ctx");
  if (!pos || !noise_emb || !out || (ctx > 0 && !taps)) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (!aligned16(noise_emb) || !aligned16(out) || (ctx > 0 && !aligned16(taps)))
    return fail(DFLASH_ERR_INVALID_ARG, "taps / noise_emb / out must start on a 16-byte boundary");
  if (ctx + kBlock > h->cfg.max_seq_len) return fail(DFLASH_ERR_CAPACITY, "ctx exceeds max_seq_len");
  {
    // the static region is looked up on the current device and bound to the
    // handle at its first use: only the handle's own device may call
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device)
      return fail(DFLASH_ERR_INVALID_ARG, "the current device (%d) is not the handle's device (%d)", dev, h->device);
  }
  // one page of K (or V^T) for every layer, with its row scales for e4m3
  const size_t page_bytes = (size_t)h->g.L * h->g.Hkv * kPage *
                            ((size_t)h->g.d * esize_kv(h->cfg.kv_dtype) + (h->attn_fp8 ? 4 : 0));
  const int fixed_pages = (int)(kFixedKvBytes / (2 * page_bytes));
  const int need = (ctx + kBlock + kPage - 1) / kPage;
  if (need > fixed_pages)
    return fail(DFLASH_ERR_CAPACITY, "ctx %d exceeds the static KV region (at most %d context rows for this drafter)",
                ctx, std::max(0, fixed_pages * kPage - kBlock));
  void* base = nullptr;
  bool fresh = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    const cudaError_t e = fixed_kv_region(&base, h->uid, &fresh);
    if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "static KV region lookup: %s", cudaGetErrorString(e));
  }
  if (fresh) {
    // another handle wrote the region last: clear this drafter's K and V
    // areas before anything else can fail (the lookup already recorded this
    // handle as the region's user; a failed clear hands the region back)
    const cudaError_t e = cudaMemsetAsync(base, 0, 2 * (size_t)fixed_pages * page_bytes, s);
    if (e != cudaSuccess) {
      bool unused = false;
      fixed_kv_region(&base, 0, &unused);
      return fail(DFLASH_ERR_CUDA, "static KV region clear: %s", cudaGetErrorString(e));
    }
  }
  if (!h->fixed.kpool) {
    const int rc = guarded([&]() -> int {
      dflash_handle::KvRegion r;
      r.kpool = static_cast<char*>(base);
      r.vpool = r.kpool + (size_t)fixed_pages * page_bytes;
      r.max_pages = fixed_pages;
      if (h->attn_tc) {
        const uint64_t rows = (uint64_t)h->g.L * fixed_pages * h->g.Hkv;
        if (h->attn_fp8) {
          kv_maps_fp8(r, r.kpool, r.vpool, rows, h->g.d);
        } else {
          r.kmap = make_map_bf16(r.kpool, rows * kPage, h->g.d, kPage);
          r.vmap = make_map_bf16(r.vpool, rows * h->g.d, kPage, h->g.d);
        }
      }
      h->fixed = std::move(r);
      return DFLASH_OK;
    });
    if (rc != DFLASH_OK) return rc;
  }
  release_slot(h, h->cfg.max_seqs);   // pool pages, if any were left
  h->fixed.free_pages.resize(h->fixed.max_pages);
  for (int i = 0; i < h->fixed.max_pages; ++i) h->fixed.free_pages[i] = h->fixed.max_pages - 1 - i;
  RegionScope scope(h, &h->fixed);
  return first_light(h, ctx, taps, noise_emb, pos, out, s);
}

int dflash_set_ctx_cap(dflash_t* h, int32_t cap) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (cap < 0) return fail(DFLASH_ERR_INVALID_ARG, "negative context cap");
  h->ctx_cap = cap;
  for (int slot = 0; slot < h->cfg.max_seqs; ++slot) evict_window(h, slot);
  return DFLASH_OK;
}

int dflash_seq_reset(dflash_t* h, int32_t seq_id) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (seq_id < 0 || seq_id >= h->cfg.max_seqs) return fail(DFLASH_ERR_INVALID_ARG, "seq id %d out of range", seq_id);
  release_slot(h, seq_id);
  return DFLASH_OK;
}

int dflash_seq_len(dflash_t* h, int32_t seq_id, int64_t* len) {
  g_last_error.clear();
  if (!h || !len) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (seq_id < 0 || seq_id >= h->cfg.max_seqs) return fail(DFLASH_ERR_INVALID_ARG, "seq id %d out of range", seq_id);
  *len = h->len[seq_id];
  return DFLASH_OK;
}

// ---------------------------------------------------------------- draft tokens
static size_t lm_blocks_bytes(const dflash_t* h, int32_t vocab) {
  return ((size_t)vocab * h->g.H * 2 + 255) / 256 * 256;
}

static int check_lm(const dflash_t* h, int32_t vocab) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (!h->use_tc) return fail(DFLASH_ERR_UNSUPPORTED, "draft tokens need bf16 or e4m3 drafter weights");
  if (vocab <= 0 || vocab % kTileN) return fail(DFLASH_ERR_INVALID_ARG, "vocab must be a positive multiple of 128");
  return DFLASH_OK;
}

int dflash_lm_head_bytes(const dflash_t* h, int32_t vocab, size_t* bytes) {
  g_last_error.clear();
  if (int rc = check_lm(h, vocab)) return rc;
  if (!bytes) return fail(DFLASH_ERR_INVALID_ARG, "bytes is null");
  *bytes = lm_blocks_bytes(h, vocab) + (size_t)h->lo.Mt * vocab * 4;
  return DFLASH_OK;
}

int dflash_pack_lm_head(dflash_t* h, const void* lm_head, int32_t vocab, void* packed, size_t bytes, void* stream) {
  g_last_error.clear();
  if (int rc = check_lm(h, vocab)) return rc;
  if (!lm_head || !packed) return fail(DFLASH_ERR_INVALID_ARG, "lm_head / packed is null");
  if (!aligned16(lm_head)) return fail(DFLASH_ERR_INVALID_ARG, "lm_head must start on a 16-byte boundary");
  if (reinterpret_cast<uintptr_t>(packed) % 256) return fail(DFLASH_ERR_INVALID_ARG, "packed must be 256-byte aligned");
  if (bytes < lm_blocks_bytes(h, vocab) + (size_t)h->lo.Mt * vocab * 4)
    return fail(DFLASH_ERR_CAPACITY, "packed buffer smaller than dflash_lm_head_bytes");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return guarded([&]() -> int {
    launch_repack(packed, h->g.H, lm_head, vocab, vocab, 0, 0, s);
    ck(cudaGetLastError(), "lm_head repack");
    return DFLASH_OK;
  });
}

int dflash_draft_tokens(dflash_t* h, int32_t n_seq, const float* hidden, const void* packed, int32_t vocab,
                        int32_t* tokens, void* stream) {
  g_last_error.clear();
  if (int rc = check_lm(h, vocab)) return rc;
  if (!hidden || !packed || !tokens) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (n_seq < 1 || n_seq > h->cfg.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "n_seq out of range");
  if (!aligned16(hidden)) return fail(DFLASH_ERR_INVALID_ARG, "hidden must start on a 16-byte boundary");
  if (reinterpret_cast<uintptr_t>(packed) % 256) return fail(DFLASH_ERR_INVALID_ARG, "packed must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n_tok = n_seq * kBlock;
  return guarded([&]() -> int {
    const Geo& g = h->g;
    float* logits = reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(packed)) + lm_blocks_bytes(h, vocab));
    {
      Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * g.H * 8, s);
      launch_to_operand(hidden, n_tok, g.H, h->at<void>(h->lo.op_h), (long)h->lo.Mt * g.H, s);
    }
    ck(cudaGetLastError(), "lm_head operand launch");
    ck(cudaMemsetAsync(logits, 0, (size_t)n_tok * vocab * 4, s), "logits clear");
    GemmSpec sp;
    sp.site = 0;
    sp.W = packed;
    sp.wscale = nullptr;
    sp.N = vocab;
    sp.K = g.H;
    sp.X = h->at<void>(h->lo.op_h);
    sp.xmap = h->xmap_h;
    sp.omode = O_RED;
    sp.dst = logits;
    sp.dst_ld = vocab;
    sp.e = base_epi(h);
    sp.e.n_tok = n_tok;
    run_gemm(h, sp, s);
    {
      Launch L(h, DFLASH_KERNEL_FINISH, (double)n_tok * vocab * 4, s);
      launch_argmax(logits, n_tok, vocab, tokens, s);
    }
    ck(cudaGetLastError(), "argmax launch");
    h->last_stream = s;
    return DFLASH_OK;
  });
}

int dflash_kv_read(dflash_t* h, int32_t seq_id, int32_t layer, int32_t row0, int32_t nrows, float* k_out,
                   float* v_out, void* stream) {
  g_last_error.clear();
  if (!h || !k_out || !v_out) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (seq_id < 0 || seq_id >= h->cfg.max_seqs) return fail(DFLASH_ERR_INVALID_ARG, "seq id %d out of range", seq_id);
  if (layer < 0 || layer >= h->cfg.n_layers) return fail(DFLASH_ERR_INVALID_ARG, "layer out of range");
  if (row0 < 0 || nrows < 0 || row0 + (int64_t)nrows > h->len[seq_id])
    return fail(DFLASH_ERR_INVALID_ARG, "rows [%d, %d) outside the %lld committed rows", row0, row0 + nrows,
                (long long)h->len[seq_id]);
  if (nrows > 0 && row0 / kPage < h->kstart[seq_id] / kPage)
    return fail(DFLASH_ERR_INVALID_ARG, "rows before %lld were evicted by the context window",
                (long long)(h->kstart[seq_id] / kPage * kPage));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return guarded([&]() -> int {
    launch_kv_read(h->g, h->at<void>(h->lo.kpool), h->at<void>(h->lo.vpool), h->at<int>(h->lo.btab), seq_id, layer,
                   row0, nrows, k_out, v_out, s);
    ck(cudaGetLastError(), "kv read launch");
    return DFLASH_OK;
  });
}

int dflash_device_status(dflash_t* h, void* stream) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  return guarded([&]() -> int {
    int err = 0;
    cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : h->last_stream;
    ck(cudaMemcpyAsync(&err, h->ws + h->lo.err, 4, cudaMemcpyDeviceToHost, s), "error word read");
    ck(cudaStreamSynchronize(s), "status sync");
    if (err) {
      // reported once: the word is cleared for the calls that follow
      ck(cudaMemsetAsync(h->ws + h->lo.err, 0, 4, s), "error word clear");
      ck(cudaStreamSynchronize(s), "status sync");
    }
    if (err == DERR_TIMEOUT) return fail(DFLASH_ERR_TIMEOUT, "a device-side wait timed out");
    if (err) return fail(DFLASH_ERR_CUDA, "device error word %d", err);
    return DFLASH_OK;
  });
}

int dflash_selftest_wait_timeout(dflash_t* h, int32_t limit_ms, void* stream) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (limit_ms < 1 || limit_ms > 2000) return fail(DFLASH_ERR_INVALID_ARG, "limit_ms must be 1..2000");
  return guarded([&]() -> int {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_selftest_wait(h->at<int>(h->lo.err), (unsigned long long)limit_ms * 1000000ull, s);
    ck(cudaGetLastError(), "self-test launch");
    h->last_stream = s;
    return DFLASH_OK;
  });
}

int dflash_profile_enable(dflash_t* h, int32_t enable) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  return guarded([&]() -> int {
    if (!h->recs.empty()) ck(cudaDeviceSynchronize(), "profile sync");
    for (auto& r : h->recs) {
      h->event_pool.push_back(r.a);
      h->event_pool.push_back(r.b);
    }
    h->recs.clear();
    h->prof_on = enable != 0;
    return DFLASH_OK;
  });
}

int dflash_profile_read(dflash_t* h, int32_t kind, int64_t* launches, double* ms, double* bytes) {
  g_last_error.clear();
  if (!h || !launches || !ms || !bytes) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (kind < 0 || kind >= DFLASH_KERNEL_KINDS) return fail(DFLASH_ERR_INVALID_ARG, "unknown kernel kind %d", kind);
  return guarded([&]() -> int {
    *launches = 0;
    *ms = 0;
    *bytes = 0;
    for (auto& r : h->recs) {
      if (r.kind != kind) continue;
      ck(cudaEventSynchronize(r.b), "profile event sync");
      float t = 0;
      ck(cudaEventElapsedTime(&t, r.a, r.b), "profile elapsed");
      *launches += 1;
      *ms += t;
      *bytes += r.bytes;
    }
    return DFLASH_OK;
  });
}

int dflash_trace_begin(dflash_t* h, void* device_buffer, size_t bytes) {
  g_last_error.clear();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is null");
  if (device_buffer && reinterpret_cast<uintptr_t>(device_buffer) % 8)
    return fail(DFLASH_ERR_INVALID_ARG, "trace buffer must be 8-byte aligned");
  if (!h->traced_execs.empty()) {
    cudaDeviceSynchronize();
    for (auto e : h->traced_execs) cudaGraphExecDestroy(e);
    h->traced_execs.clear();
  }
  h->trace_buf = static_cast<unsigned long long*>(device_buffer);
  h->trace_cap = device_buffer ? bytes / 8 : 0;
  h->trace_used = 0;
  h->trace_recs.clear();
  return DFLASH_OK;
}

int dflash_trace_launches(dflash_t* h, int32_t max_launches, int32_t* kinds, int32_t* grids, int64_t* offsets,
                          int32_t* n_launches) {
  g_last_error.clear();
  if (!h || !n_launches) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  const int n = (int)h->trace_recs.size();
  *n_launches = n;
  for (int i = 0; i < n && i < max_launches; ++i) {
    if (kinds) kinds[i] = h->trace_recs[i].kind;
    if (grids) grids[i] = h->trace_recs[i].grid;
    if (offsets) offsets[i] = h->trace_recs[i].offset;
  }
  return DFLASH_OK;
}

int dflash_launch_count(dflash_t* h, int64_t* launches) {
  g_last_error.clear();
  if (!h || !launches) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  *launches = h->launches;
  return DFLASH_OK;
}

void dflash_destroy(dflash_t* h) {
  if (!h) return;
  for (auto& r : h->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : h->event_pool) cudaEventDestroy(e);
  for (auto& gr : h->graphs) {
    cudaGraphExecDestroy(gr.exec);
    cudaGraphDestroy(gr.graph);
  }
  if (!h->traced_execs.empty()) cudaDeviceSynchronize();
  for (auto e : h->traced_execs) cudaGraphExecDestroy(e);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  delete h;
}

}  // extern "C"
