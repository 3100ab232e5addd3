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

int esize_w(int wtype) { return wtype == DFLASH_F32 ? 4 : (wtype == DFLASH_BF16 ? 2 : 1); }
int esize_kv(int kvtype) { return kvtype == DFLASH_F32 ? 4 : 2; }

// Workspace carve-up, computed identically by dflash_workspace_bytes and dflash_create.
struct Layout {
  size_t fc, qkv, o, gu, down, kvall;                   // weights
  size_t s_fc, s_qkv, s_o, s_gu, s_down, s_kvall;       // fp8 row scales
  size_t hn, fn, in_ln, post_ln, qn, kn;                // norm gains
  size_t kpool, vpool, btab, inv_freq;
  size_t h, op_h, op_taps, op_o, op_a, q, ss;
  size_t part, counters, apart_o, apart_ml, rdesc, idesc, err;
  size_t total;
  int Mt, pps, max_tiles, grid_max, items_cap, n_sites;
};

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
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
  Lo.items_cap = 2 * n_sm + (int)Hkv * c.max_batch;
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
  Lo.kpool = take(L * (size_t)c.max_pages * Hkv * kPage * d * ek);
  Lo.vpool = take(L * (size_t)c.max_pages * Hkv * kPage * d * ek);
  Lo.btab = take((size_t)(c.max_seqs + 1) * Lo.pps * 4);
  Lo.inv_freq = take(d / 2 * 8);
  Lo.h = take(Mt * H * 4);
  Lo.op_h = take(Mt * H * 4);
  Lo.op_taps = take(Mt * nH * 4);
  Lo.op_o = take(Mt * Hq * d * 4);
  Lo.op_a = take(Mt * I * 4);
  Lo.q = take(Mt * Hq * d * 4);
  Lo.ss = take((2 * L + 2) * Mt * 4);
  Lo.part = take((size_t)(Lo.grid_max + Lo.max_tiles) * Mt * kTileN * 4);
  Lo.counters = take((size_t)Lo.n_sites * Lo.max_tiles * 4);
  Lo.apart_o = take((size_t)Lo.items_cap * R * d * 4);
  Lo.apart_ml = take((size_t)Lo.items_cap * R * 2 * 4);
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
  if (c->kv_dtype != DFLASH_F32 && c->kv_dtype != DFLASH_BF16) return fail(DFLASH_ERR_INVALID_ARG, "kv_dtype");
  if (c->weight_dtype == DFLASH_F32 && c->kv_dtype != DFLASH_F32)
    return fail(DFLASH_ERR_UNSUPPORTED, "f32 weights need an f32 KV cache");
  if (c->weight_dtype != DFLASH_F32 && c->kv_dtype != DFLASH_BF16)
    return fail(DFLASH_ERR_UNSUPPORTED, "bf16/fp8 weights need a bf16 KV cache");
  if (c->rope_type != DFLASH_ROPE_PLAIN && c->rope_type != DFLASH_ROPE_YARN) return fail(DFLASH_ERR_INVALID_ARG, "rope_type");
  if (!(c->rope_theta > 1.0)) return fail(DFLASH_ERR_INVALID_ARG, "rope_theta must be > 1");
  if (c->rope_type == DFLASH_ROPE_YARN &&
      (!(c->yarn_factor >= 1.0) || c->yarn_original_max_pos < 1 || !(c->yarn_beta_fast > 0) || !(c->yarn_beta_slow > 0)))
    return fail(DFLASH_ERR_INVALID_ARG, "bad YaRN parameters");
  if (!(c->rms_eps > 0)) return fail(DFLASH_ERR_INVALID_ARG, "rms_eps must be > 0");
  if (c->max_seqs < 1 || c->max_pages < 1 || c->max_seq_len < kBlock + 1)
    return fail(DFLASH_ERR_INVALID_ARG, "capacity fields must be positive");
  if (c->max_batch < 1 || c->max_batch > kMaxBatch) return fail(DFLASH_ERR_INVALID_ARG, "max_batch must be 1..64");
  if (c->max_ingest_rows < 1 || c->max_ingest_rows > kMaxIngestRows)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ingest_rows must be 1..512");
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

}  // namespace

struct dflash_handle {
  dflash_config cfg;
  Layout lo;
  char* ws;
  Geo g;
  int n_sm;
  std::vector<int64_t> len;               // committed rows per slot (slot max_seqs = internal)
  std::vector<std::vector<int>> pages;    // page ids per slot
  std::vector<int> free_pages;
  cudaStream_t last_stream = nullptr;
  // measurement: kernel launches issued, and (when enabled) per-kind event pairs
  int64_t launches = 0;
  // tensor maps of the tensor-core projections: weights per GEMM site, operands per buffer
  std::vector<CUtensorMap> wmap;
  CUtensorMap xmap_taps, xmap_h, xmap_o, xmap_a;
  bool use_tc = false;
  bool prof_on = false;
  struct Rec {
    int kind;
    cudaEvent_t a, b;
    double bytes;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> event_pool;
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

// Reserve pages so that slot covers `rows` rows; records block-table entries.
bool ensure_pages(dflash_t* h, int slot, int64_t rows, InitBlob& blob, std::vector<int>& taken) {
  const int need = (int)((rows + kPage - 1) / kPage);
  auto& pl = h->pages[slot];
  while ((int)pl.size() < need) {
    if (h->free_pages.empty() || blob.n_pt >= kMaxPtUpdates) return false;
    const int page = h->free_pages.back();
    h->free_pages.pop_back();
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
    h->free_pages.push_back(pl.back());
    pl.pop_back();
  }
  (void)blob;
}

EpiArgs base_epi(dflash_t* h) {
  EpiArgs e{};
  e.g = h->g;
  e.inv_freq = h->at<double>(h->lo.inv_freq);
  e.block_table = h->at<int>(h->lo.btab);
  e.kpool = h->at<void>(h->lo.kpool);
  e.vpool = h->at<void>(h->lo.vpool);
  e.rd = h->at<RoundDesc>(h->lo.rdesc);
  e.id = h->at<IngestDesc>(h->lo.idesc);
  e.err = h->at<int>(h->lo.err);
  e.op_f32 = h->cfg.weight_dtype == DFLASH_F32;
  return e;
}

// One projection: passes of <= 256 token columns; tensor cores for bf16
// weights, CUDA cores for f32 weights (and, for now, fp8 weights).
void run_gemm(dflash_t* h, int site, const void* W, const float* wscale, int N, int K, const void* X,
              const CUtensorMap* xmap, EpiArgs e, cudaStream_t s) {
  const Geo& g = h->g;
  const int n_all = e.n_tok;
  for (int base = 0; base < n_all; base += 256) {
    GemmArgs a{};
    a.W = W;
    a.N = N;
    a.K = K;
    a.X = X;
    a.x_ld = K;
    a.x_plane = (long)h->lo.Mt * K;
    a.x_f32 = h->cfg.weight_dtype == DFLASH_F32;
    a.n_tiles = N / kTileN;
    a.p.kb = K / kTileK;
    a.p.units = a.n_tiles * a.p.kb;
    a.p.grid = std::min(a.p.units, h->use_tc ? h->n_sm : h->lo.grid_max);
    a.part = h->at<float>(h->lo.part);
    a.counters = h->at<int>(h->lo.counters) + (size_t)site * h->lo.max_tiles;
    e.wscale = wscale;
    e.tok_base = base;
    e.n_tok = std::min(256, n_all - base);
    a.e = e;
    const double nt = e.n_tok;
    double out_b = 0;
    switch (e.kind) {
      case EPI_FC: out_b = nt * N * 4; break;
      case EPI_KV: out_b = nt * N * (g.kvtype == KV_F32 ? 4 : 2); break;
      case EPI_QKV: out_b = nt * N * (g.kvtype == KV_F32 ? 4 : 2); break;
      case EPI_RESID: out_b = nt * N * 12; break;
      default: out_b = nt * N / 2 * 4; break;
    }
    const double bytes =
        (double)N * K * esize_w(g.wtype) + (g.wtype == W_FP8 ? N * 4.0 : 0.0) + nt * K * 4 + out_b;
    Launch L(h, DFLASH_KERNEL_GEMM, bytes, s);
    if (h->use_tc) launch_gemm_tc(a, &h->wmap[site], xmap, s);
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
  ia.op = h->at<void>(h->lo.op_taps);
  ia.op_ld = width;
  ia.op_plane = (long)h->lo.Mt * width;
  ia.op_f32 = h->cfg.weight_dtype == DFLASH_F32;
  float* ss_feat = h->at<float>(h->lo.ss) + (size_t)(2 * g.L + 1) * h->lo.Mt;
  ia.zero_ptr = ss_feat;
  ia.zero_n = n_rows;
  ia.desc_dst = h->at<void>(h->lo.idesc);
  ia.desc_bytes = sizeof(IngestDesc);
  ia.block_table = h->at<int>(h->lo.btab);
  ia.g = g;
  {
    Launch L(h, DFLASH_KERNEL_INIT, (double)n_rows * width * 8, s);
    launch_init(ia, blob, s);
  }
  ck(cudaGetLastError(), "ingest init launch");

  // fc over the taps; epilogue: feats operand (c * hidden_norm) + sum c^2
  EpiArgs e = base_epi(h);
  e.kind = EPI_FC;
  e.n_tok = n_rows;
  e.ss_out = ss_feat;
  e.gain = h->at<float>(h->lo.hn);
  e.op = h->at<void>(h->lo.op_h);
  e.op_ld = g.H;
  e.op_plane = (long)h->lo.Mt * g.H;
  const bool fp8 = h->cfg.weight_dtype == DFLASH_FP8_E4M3;
  run_gemm(h, 0, h->at<void>(h->lo.fc), fp8 ? h->at<float>(h->lo.s_fc) : nullptr, g.H, width,
           h->at<void>(h->lo.op_taps), &h->xmap_taps, e, s);

  // K/V of every layer in one projection; epilogue: hidden_norm scale,
  // k head-norm + RoPE, paged write.
  EpiArgs k = base_epi(h);
  k.kind = EPI_KV;
  k.n_tok = n_rows;
  k.ss_in = ss_feat;
  k.kn = h->at<float>(h->lo.kn);
  run_gemm(h, 1, h->at<void>(h->lo.kvall), fp8 ? h->at<float>(h->lo.s_kvall) : nullptr, g.L * g.kv_n, g.H,
           h->at<void>(h->lo.op_h), &h->xmap_h, k, s);
}

int choose_split_pages(dflash_t* h, const std::vector<int64_t>& lens) {
  long units = 0;
  for (auto L : lens) units += (long)h->g.Hkv * ((L + kBlock + kPage - 1) / kPage);
  const long target = 2L * h->n_sm;
  return (int)std::max<long>(1, (units + target - 1) / target);
}

void enqueue_round(dflash_t* h, InitBlob& blob, const float* noise, float* out, cudaStream_t s) {
  const Geo& g = h->g;
  RoundDesc& rd = blob.round;
  const int n_tok = rd.n_tok;
  const size_t Mt = h->lo.Mt;
  float* ss = h->at<float>(h->lo.ss);
  auto ss_in = [&](int l) { return ss + (size_t)l * Mt; };
  auto ss_post = [&](int l) { return ss + (size_t)(g.L + l) * Mt; };
  float* ss_fin = ss + (size_t)(2 * g.L) * Mt;
  const bool fp8 = h->cfg.weight_dtype == DFLASH_FP8_E4M3;
  const size_t ew = wbytes(h);

  InitArgs ia{};
  ia.src = noise;
  ia.n_rows = n_tok;
  ia.width = g.H;
  ia.h = h->at<float>(h->lo.h);
  ia.ss0 = ss_in(0);
  ia.gain = h->at<float>(h->lo.in_ln);
  ia.op = h->at<void>(h->lo.op_h);
  ia.op_ld = g.H;
  ia.op_plane = (long)Mt * g.H;
  ia.op_f32 = h->cfg.weight_dtype == DFLASH_F32;
  ia.zero_ptr = ss + Mt;                    // every per-token accumulator after ss_in(0)
  ia.zero_n = (int)((2 * g.L + 1 - 1) * Mt);
  ia.desc_dst = h->at<void>(h->lo.rdesc);
  ia.desc_bytes = sizeof(RoundDesc);
  ia.block_table = h->at<int>(h->lo.btab);
  ia.g = g;
  {
    Launch L(h, DFLASH_KERNEL_INIT, (double)n_tok * g.H * 12, s);
    launch_init(ia, blob, s);
  }
  ck(cudaGetLastError(), "round init launch");

  for (int l = 0; l < g.L; ++l) {
    // QKV: epilogue = input-norm scale, q/k head-norm + RoPE, block K/V into the pages
    EpiArgs e = base_epi(h);
    e.kind = EPI_QKV;
    e.layer = l;
    e.n_tok = n_tok;
    e.ss_in = ss_in(l);
    e.qn = h->at<float>(h->lo.qn) + (size_t)l * g.d;
    e.kn = h->at<float>(h->lo.kn) + (size_t)l * g.d;
    e.q_out = h->at<void>(h->lo.q);
    run_gemm(h, 2 + 4 * l, h->at<char>(h->lo.qkv) + (size_t)l * g.qkv_n * g.H * ew,
             fp8 ? h->at<float>(h->lo.s_qkv) + (size_t)l * g.qkv_n : nullptr, g.qkv_n, g.H,
             h->at<void>(h->lo.op_h), &h->xmap_h, e, s);

    // attention over [cached ctx ; block] K/V, split over keys, then merge
    AttnArgs a{};
    a.q = h->at<void>(h->lo.q);
    a.kpool = h->at<void>(h->lo.kpool);
    a.vpool = h->at<void>(h->lo.vpool);
    a.layer = l;
    a.block_table = h->at<int>(h->lo.btab);
    a.rd = h->at<RoundDesc>(h->lo.rdesc);
    a.part_o = h->at<float>(h->lo.apart_o);
    a.part_ml = h->at<float>(h->lo.apart_ml);
    a.op = h->at<void>(h->lo.op_o);
    a.op_ld = g.Hq * g.d;
    a.op_plane = (long)Mt * g.Hq * g.d;
    a.op_f32 = h->cfg.weight_dtype == DFLASH_F32;
    a.scale = 1.f / std::sqrt((float)g.d);
    a.err = h->at<int>(h->lo.err);
    a.g = g;
    const double ekv = g.kvtype == KV_F32 ? 4 : 2;
    const double part_b = (double)rd.n_items * g.G * kBlock * (g.d + 2) * 4;
    {
      double kv_b = 0;
      for (int i = 0; i < rd.n_seq; ++i) kv_b += (double)(rd.len[i] + kBlock) * g.Hkv * g.d * 2 * ekv;
      Launch L(h, DFLASH_KERNEL_ATTENTION, kv_b + (double)n_tok * g.Hq * g.d * ekv + part_b, s);
      launch_attention_simt(a, rd.n_items, s);
    }
    ck(cudaGetLastError(), "attention launch");
    {
      Launch L(h, DFLASH_KERNEL_COMBINE, part_b + (double)n_tok * g.Hq * g.d * 4, s);
      launch_attn_combine(a, n_tok, s);
    }
    ck(cudaGetLastError(), "attention combine launch");

    // O projection + residual; operand for the MLP = h * post_ln
    EpiArgs o = base_epi(h);
    o.kind = EPI_RESID;
    o.n_tok = n_tok;
    o.h = h->at<float>(h->lo.h);
    o.h_ld = g.H;
    o.gain = h->at<float>(h->lo.post_ln) + (size_t)l * g.H;
    o.ss_out = ss_post(l);
    o.op = h->at<void>(h->lo.op_h);
    o.op_ld = g.H;
    o.op_plane = (long)Mt * g.H;
    run_gemm(h, 3 + 4 * l, h->at<char>(h->lo.o) + (size_t)l * g.H * g.Hq * g.d * ew,
             fp8 ? h->at<float>(h->lo.s_o) + (size_t)l * g.H : nullptr, g.H, g.Hq * g.d,
             h->at<void>(h->lo.op_o), &h->xmap_o, o, s);

    // gate/up (interleaved per 64 rows) + SwiGLU
    EpiArgs gu = base_epi(h);
    gu.kind = EPI_SWIGLU;
    gu.n_tok = n_tok;
    gu.ss_in = ss_post(l);
    gu.op = h->at<void>(h->lo.op_a);
    gu.op_ld = g.I;
    gu.op_plane = (long)Mt * g.I;
    run_gemm(h, 4 + 4 * l, h->at<char>(h->lo.gu) + (size_t)l * 2 * g.I * g.H * ew,
             fp8 ? h->at<float>(h->lo.s_gu) + (size_t)l * 2 * g.I : nullptr, 2 * g.I, g.H,
             h->at<void>(h->lo.op_h), &h->xmap_h, gu, s);

    // down + residual; operand for the next layer = h * input_ln[l+1]
    EpiArgs dn = base_epi(h);
    dn.kind = EPI_RESID;
    dn.n_tok = n_tok;
    dn.h = h->at<float>(h->lo.h);
    dn.h_ld = g.H;
    const bool last = l + 1 == g.L;
    dn.gain = last ? nullptr : h->at<float>(h->lo.in_ln) + (size_t)(l + 1) * g.H;
    dn.ss_out = last ? ss_fin : ss_in(l + 1);
    dn.op = last ? nullptr : h->at<void>(h->lo.op_h);
    dn.op_ld = g.H;
    dn.op_plane = (long)Mt * g.H;
    run_gemm(h, 5 + 4 * l, h->at<char>(h->lo.down) + (size_t)l * g.H * g.I * ew,
             fp8 ? h->at<float>(h->lo.s_down) + (size_t)l * g.H : nullptr, g.H, g.I,
             h->at<void>(h->lo.op_a), &h->xmap_a, dn, s);
  }
  {
    Launch L(h, DFLASH_KERNEL_NORM, (double)n_tok * g.H * 8, s);
    launch_final_norm(h->at<float>(h->lo.h), ss_fin, h->at<float>(h->lo.fn), out, n_tok, g, s);
  }
  ck(cudaGetLastError(), "final norm launch");
}

// Fill the attention split plan of a round descriptor.
void plan_attention(dflash_t* h, RoundDesc& rd, const std::vector<int64_t>& lens) {
  rd.split_pages = choose_split_pages(h, lens);
  int items = 0;
  for (int s = 0; s < rd.n_seq; ++s) {
    rd.item0[s] = items;
    const int pages = (int)((lens[s] + kBlock + kPage - 1) / kPage);
    items += h->g.Hkv * ((pages + rd.split_pages - 1) / rd.split_pages);
  }
  rd.item0[rd.n_seq] = items;
  rd.n_items = items;
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
      id.row_slot[r] = slot;
      id.row_dst[r] = (int)h->len[slot] + j;
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
  for (int i = 0; i < n_seq; ++i) h->len[slots[i]] += t_per_seq[i];
  h->last_stream = s;
  delete blob;
  return DFLASH_OK;
}

int round_slots(dflash_t* h, int n_seq, const int32_t* slots, const int32_t* pos_block, const float* noise,
                float* out, cudaStream_t s) {
  if (!pos_block || !noise || !out) return fail(DFLASH_ERR_INVALID_ARG, "pos_block / noise_emb / out is null");
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
    for (int j = 0; j < kBlock; ++j) rd.pos[i * kBlock + j] = pos_block[i * kBlock + j];
    if (!ensure_pages(h, slot, lens[i] + kBlock, *blob, taken)) {
      rollback_pages(h, *blob, taken);
      delete blob;
      return fail(DFLASH_ERR_CAPACITY, "out of KV pages for the block rows");
    }
  }
  plan_attention(h, rd, lens);
  if (rd.n_items > h->lo.items_cap) {
    rollback_pages(h, *blob, taken);
    delete blob;
    return fail(DFLASH_ERR_CAPACITY, "attention plan exceeds its scratch");
  }
  int rc = guarded([&]() -> int {
    enqueue_round(h, *blob, noise, out, s);
    return DFLASH_OK;
  });
  if (rc != DFLASH_OK) rollback_pages(h, *blob, taken);
  else h->last_stream = s;
  delete blob;
  return rc;
}

void release_slot(dflash_t* h, int slot) {
  for (int p : h->pages[slot]) h->free_pages.push_back(p);
  h->pages[slot].clear();
  h->len[slot] = 0;
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
  }
  const int n_sm = sm_count();
  Layout lo = make_layout(*cfg, n_sm);
  if (ws_bytes < lo.total) return fail(DFLASH_ERR_CAPACITY, "workspace %zu bytes < required %zu", ws_bytes, lo.total);

  dflash_t* h = new (std::nothrow) dflash_handle();
  if (!h) return fail(DFLASH_ERR_CAPACITY, "host allocation failed");
  h->cfg = *cfg;
  h->lo = lo;
  h->ws = static_cast<char*>(workspace);
  h->n_sm = n_sm;
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
  h->free_pages.resize(cfg->max_pages);
  for (int i = 0; i < cfg->max_pages; ++i) h->free_pages[i] = cfg->max_pages - 1 - i;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = guarded([&]() -> int {
    const size_t ew = esize_w(cfg->weight_dtype);
    auto cp = [&](size_t dst_off, const void* src, size_t bytes) {
      ck(cudaMemcpyAsync(h->ws + dst_off, src, bytes, cudaMemcpyDeviceToDevice, s), "weight copy");
    };
    cp(lo.fc, w->fc, (size_t)H * g.n * H * ew);
    if (fp8) cp(lo.s_fc, w->fc_scale, (size_t)H * 4);
    cp(lo.hn, w->hidden_norm, (size_t)H * 4);
    cp(lo.fn, w->norm, (size_t)H * 4);
    for (int l = 0; l < L; ++l) {
      const dflash_layer_weights& W = w->layers[l];
      const size_t qr = (size_t)Hq * d, kr = (size_t)Hkv * d;
      const size_t qkv0 = lo.qkv + (size_t)l * g.qkv_n * H * ew;
      cp(qkv0, W.q, qr * H * ew);
      cp(qkv0 + qr * H * ew, W.k, kr * H * ew);
      cp(qkv0 + (qr + kr) * H * ew, W.v, kr * H * ew);
      const size_t kv0 = lo.kvall + (size_t)l * g.kv_n * H * ew;
      cp(kv0, W.k, kr * H * ew);
      cp(kv0 + kr * H * ew, W.v, kr * H * ew);
      cp(lo.o + (size_t)l * H * Hq * d * ew, W.o, (size_t)H * Hq * d * ew);
      cp(lo.down + (size_t)l * H * I * ew, W.down, (size_t)H * I * ew);
      // gate/up interleaved in blocks of 64 rows: [g0..63, u0..63, g64..127, u64..127, ...]
      const size_t blk = (size_t)64 * H * ew;
      const size_t gu0 = lo.gu + (size_t)l * 2 * I * H * ew;
      ck(cudaMemcpy2DAsync(h->ws + gu0, 2 * blk, W.gate, blk, blk, I / 64, cudaMemcpyDeviceToDevice, s), "gate copy");
      ck(cudaMemcpy2DAsync(h->ws + gu0 + blk, 2 * blk, W.up, blk, blk, I / 64, cudaMemcpyDeviceToDevice, s), "up copy");
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
    h->use_tc = cfg->weight_dtype == DFLASH_BF16;
    if (h->use_tc) {
      const uint64_t Mt2 = 2ull * lo.Mt;
      h->wmap.resize(lo.n_sites);
      h->wmap[0] = make_map_bf16(h->ws + lo.fc, H, (uint64_t)g.n * H, kTileN);
      h->wmap[1] = make_map_bf16(h->ws + lo.kvall, (uint64_t)L * g.kv_n, H, kTileN);
      for (int l = 0; l < L; ++l) {
        h->wmap[2 + 4 * l] = make_map_bf16(h->ws + lo.qkv + (size_t)l * g.qkv_n * H * 2, g.qkv_n, H, kTileN);
        h->wmap[3 + 4 * l] = make_map_bf16(h->ws + lo.o + (size_t)l * H * Hq * d * 2, H, (uint64_t)Hq * d, kTileN);
        h->wmap[4 + 4 * l] = make_map_bf16(h->ws + lo.gu + (size_t)l * 2 * I * H * 2, 2ull * I, H, kTileN);
        h->wmap[5 + 4 * l] = make_map_bf16(h->ws + lo.down + (size_t)l * H * I * 2, H, I, kTileN);
      }
      h->xmap_taps = make_map_bf16(h->ws + lo.op_taps, Mt2, (uint64_t)g.n * H, 16);
      h->xmap_h = make_map_bf16(h->ws + lo.op_h, Mt2, H, 16);
      h->xmap_o = make_map_bf16(h->ws + lo.op_o, Mt2, (uint64_t)Hq * d, 16);
      h->xmap_a = make_map_bf16(h->ws + lo.op_a, Mt2, I, 16);
    }
    ck(cudaMemsetAsync(h->ws + lo.btab, 0xff, (size_t)(cfg->max_seqs + 1) * lo.pps * 4, s), "block table");
    ck(cudaMemsetAsync(h->ws + lo.counters, 0, (size_t)lo.n_sites * lo.max_tiles * 4, s), "counters");
    ck(cudaMemsetAsync(h->ws + lo.err, 0, 256, s), "error word");
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
  if (ctx + kBlock > h->cfg.max_seq_len) return fail(DFLASH_ERR_CAPACITY, "ctx exceeds max_seq_len");
  const int need = (ctx + kBlock + kPage - 1) / kPage;
  if ((int)h->free_pages.size() < need) return fail(DFLASH_ERR_CAPACITY, "out of KV pages");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int slot = h->cfg.max_seqs;
  release_slot(h, slot);
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

int dflash_kv_read(dflash_t* h, int32_t seq_id, int32_t layer, int32_t row0, int32_t nrows, float* k_out,
                   float* v_out, void* stream) {
  g_last_error.clear();
  if (!h || !k_out || !v_out) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (seq_id < 0 || seq_id >= h->cfg.max_seqs) return fail(DFLASH_ERR_INVALID_ARG, "seq id %d out of range", seq_id);
  if (layer < 0 || layer >= h->cfg.n_layers) return fail(DFLASH_ERR_INVALID_ARG, "layer out of range");
  if (row0 < 0 || nrows < 0 || row0 + (int64_t)nrows > h->len[seq_id])
    return fail(DFLASH_ERR_INVALID_ARG, "rows [%d, %d) outside the %lld committed rows", row0, row0 + nrows,
                (long long)h->len[seq_id]);
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
    if (err == DERR_TIMEOUT) return fail(DFLASH_ERR_TIMEOUT, "a device-side wait timed out");
    if (err) return fail(DFLASH_ERR_CUDA, "device error word %d", err);
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
  delete h;
}

}  // extern "C"
