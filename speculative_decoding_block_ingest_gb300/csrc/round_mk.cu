// round_mk.cu -- every layer of a drafting round (DflashDraft, item
// forward_round) as one persistent kernel, for rounds of up to 64 block rows.
//
// One CTA per SM, all co-resident (cooperative launch).  Dependent steps do
// not meet at kernel boundaries: each step publishes its results through
// device-wide counters and each consumer waits on exactly the counters it
// needs (a projection tile, a kv head's rows, a split group, an activation
// block, the residual rows).  Weight blocks depend on nothing, so they stream
// through a ring of shared-memory stages continuously, across projections and
// layers, while the CTA waits for data.
//
// Warps (8 x 32 threads):
//   0     weight producer: every projection unit's 16 KB block, in order;
//   1     MMA issuer: the projection units and this CTA's attention item;
//   2..5  compute: accumulator drains (red.add into token-major sums), row
//         norms, q/k head norm + RoPE, softmax, split combine, SwiGLU;
//   6     attention loader: cached-context pages (ahead of their layer's
//         dependencies), then the query tile and the block-row pages;
//   7     operand producer: each unit's operand slice once its rows are final.
// Per layer: norm(h) -> QKV -> q/k finish -> attention -> combine -> O (+= h)
// -> norm(h) -> gate/up -> SwiGLU -> down (+= h); then the final norm.
#include <algorithm>
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kMkThreads = 256;
constexpr int kMkCompute = 128;          // warps 2..5
constexpr int kMkBar = 2;                // named barrier of the compute warps
constexpr int kMkKvStages = 2;
constexpr int kWBlk = kTileN * kTileK * 2;   // 16 KB weight block
constexpr int kQAtom = 128 * 128;            // 128 rows x 128 B
constexpr int kKAtom = 64 * 128;             // 64 keys x 128 B
constexpr int kPBytes = 128 * 128;           // P tile: 128 rows x 64 keys bf16
constexpr float kRescaleLog2 = 8.f;
constexpr int kMkRowVec = kMaxHidden / (4 * kMkCompute);   // float4 per compute thread

__device__ __forceinline__ void mk_sync() {
  asm volatile("barrier.sync %0, %1;" ::"r"(kMkBar), "r"(kMkCompute) : "memory");
}

struct MkGemm {
  const uint8_t* W;
  Part p;
  float* dst;
  int dst_ld;
};

__device__ __forceinline__ MkGemm mk_gemm(const MkArgs& a, int l, int k) {
  MkGemm m;
  if (k == 0) {
    m.W = a.wq + (size_t)l * a.wq_l;
    m.p = a.pq;
    m.dst = a.qkv_acc;
    m.dst_ld = a.g.qkv_n;
  } else if (k == 1) {
    m.W = a.wo + (size_t)l * a.wo_l;
    m.p = a.po;
    m.dst = a.h;
    m.dst_ld = a.g.H;
  } else if (k == 2) {
    m.W = a.wg + (size_t)l * a.wg_l;
    m.p = a.pg;
    m.dst = a.gu_acc;
    m.dst_ld = 2 * a.g.I;
  } else {
    m.W = a.wd + (size_t)l * a.wd_l;
    m.p = a.pd;
    m.dst = a.h;
    m.dst_ld = a.g.H;
  }
  return m;
}

__device__ __forceinline__ unsigned* mk_cnt(const MkArgs& a, int l, int off) {
  return a.cnt + (size_t)l * a.c.per_layer + off;
}

// CTAs whose stream-K range touches tile T of partition p.  With fewer
// units than CTAs some CTAs own none, so the owners of the tile's first and
// last units bound the set but are not all in it.
__device__ __forceinline__ unsigned contributors(const Part& p, int T) {
  const int lo = p.owner(T * p.kb), hi = p.owner((T + 1) * p.kb - 1);
  unsigned n = 0;
  for (int c = lo; c <= hi; ++c) n += p.start(c) < p.start(c + 1) ? 1u : 0u;
  return n;
}

// Optional trace: clock64 cycles since entry at point p (0..13) of layer l.
__device__ __forceinline__ void mk_mark(const MkArgs& a, int l, int p, unsigned long long c0) {
  if (a.trace && l < 8) {
    const unsigned long long v = trace_clock() - c0;
    asm volatile("st.global.u64 [%0], %1;" ::"l"(a.trace + (long)blockIdx.x * kMkTraceWords + 2 + 14 * l + p), "l"(v)
                 : "memory");
  }
}

__device__ __forceinline__ void raise_error(volatile int* flags, int* err) {
  flags[0] = 1;
  atomicExch(err, DERR_TIMEOUT);
}

// Thread 0 of the compute group waits; the group learns the outcome at the
// barrier (flags[0] raised on failure).
__device__ __forceinline__ void group_wait(const unsigned* c, unsigned target, volatile int* flags, int* err) {
  if (threadIdx.x == 64 && !counter_wait(c, target, flags, err)) raise_error(flags, err);
  mk_sync();
}

// Publish the group's stores, then one add: the CTA barrier orders every
// thread's stores before thread 64's release (cumulative at gpu scope).
__device__ __forceinline__ void group_signal(unsigned* c, volatile int* flags) {
  fence_proxy_async_global();
  mk_sync();
  if (threadIdx.x == 64 && !flags[0]) counter_add(c, 1);
}

// RMSNorm of one row by the 128 compute threads: out = row * gain * r.
__device__ __forceinline__ void mk_row_norm(const float* row, const float* gain, int H, float eps, float4 (&v)[kMkRowVec],
                                            float4 (&w)[kMkRowVec], float* red, int ct) {
  const int n4 = H / 4;
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const float4* g4 = reinterpret_cast<const float4*>(gain);
#pragma unroll
  for (int k = 0; k < kMkRowVec; ++k) {
    const int i = ct + k * kMkCompute;
    v[k] = i < n4 ? __ldcg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    w[k] = i < n4 ? __ldg(g4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMkRowVec; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  ss = warp_sum(ss);
  if ((ct & 31) == 0) red[ct >> 5] = ss;
  mk_sync();
  const float r = rsqrtf((red[0] + red[1] + red[2] + red[3]) / (float)H + eps);
  mk_sync();   // red is reused by the next row
#pragma unroll
  for (int k = 0; k < kMkRowVec; ++k) {
    v[k].x *= w[k].x * r;
    v[k].y *= w[k].y * r;
    v[k].z *= w[k].z * r;
    v[k].w *= w[k].w * r;
  }
}

}  // namespace

__global__ void __launch_bounds__(kMkThreads, 1)
    round_mk_kernel(const __grid_constant__ CUtensorMap tmXh, const __grid_constant__ CUtensorMap tmXo,
                    const __grid_constant__ CUtensorMap tmXa, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ MkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geo& g = a.g;
  const int S = a.stages;
  uint8_t* ring = smem;                                        // S x stage_bytes
  uint8_t* sQ = ring + (size_t)S * a.stage_bytes;              // datoms x 16 KB
  uint8_t* sP = sQ + a.datoms * kQAtom;                        // 16 KB
  uint8_t* sKV = sP + kPBytes;                                 // 2 x kv_stage_bytes
  uint8_t* ctl = sKV + kMkKvStages * a.kv_stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;                               // [2]
  uint64_t* accempty = accfull + 2;                            // [2]
  uint64_t* kvfull = accempty + 2;                             // [2]
  uint64_t* kvempty = kvfull + 2;                              // [2]
  uint64_t* sfull = kvempty + 2;                               // [2]
  uint64_t* qfull = sfull + 2;
  uint64_t* qempty = qfull + 1;
  uint64_t* pfull = qempty + 1;
  uint64_t* pvdone = pfull + 1;
  uint64_t* fin = pvdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // [0] abort
  float* red = reinterpret_cast<float*>(tmem_slot + 8);                   // [8] reductions
  float4* part4 = reinterpret_cast<float4*>(ctl + 512);                   // [128] combine partials

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, grid = gridDim.x;
  const int R = g.G * kBlock;                  // query rows of a kv head
  unsigned long long c0 = 0;
  {
    __shared__ unsigned long long c0s;
    if (threadIdx.x == 0) {
      c0s = trace_clock();
      if (a.trace) {
        unsigned smid;
        unsigned long long t;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
        a.trace[(long)c * kMkTraceWords] = smid;
        a.trace[(long)c * kMkTraceWords + 1] = t;
      }
    }
    __syncthreads();
    c0 = c0s;
  }
  const int n_tok = a.n_tok;

  // the counter set of the next round starts at zero
  for (int i = c * kMkThreads + threadIdx.x; i < a.cnt_words; i += grid * kMkThreads) a.cnt_next[i] = 0u;
  // padding rows of the query tile stay zero (the MMA reads all 128 rows)
  for (int idx = threadIdx.x; idx < a.datoms * (128 - R) * 32; idx += kMkThreads) {
    const int atom = idx / ((128 - R) * 32), rem = idx % ((128 - R) * 32);
    reinterpret_cast<uint32_t*>(sQ + atom * kQAtom + R * 128)[rem] = 0u;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);       // weight producer + operand producer
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kMkCompute);
      mbar_init(&kvfull[b], 1);
      mbar_init(&kvempty[b], 1);
      mbar_init(&sfull[b], 1);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    mbar_init(pfull, kMkCompute);
    mbar_init(pvdone, 1);
    mbar_init(fin, 1);
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmXh);
    tma_prefetch_map(&tmXo);
    tma_prefetch_map(&tmXa);
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;            // projections: cols [0, 2*aw)
  const uint32_t tatt = tmem + 256u;           // attention: O [0, d), S buffers at 128 and 192

  // this CTA's attention item (one per layer; the same item index every layer)
  const bool has_item = c < a.n_items;
  int it_s = 0, it_kvh = 0, it_k0 = 0, it_k1 = 0;
  if (has_item) attn_item(a.rd, g.Hkv, c, &it_s, &it_kvh, &it_k0, &it_k1);
  const int it_pages = (it_k1 - it_k0 + kPage - 1) / kPage;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- weight producer
      const uint64_t pol = policy_evict_first();
      int st = 0, wrap = 0;
      bool ok = true;
      for (int l = 0; l < g.L && ok; ++l)
        for (int k = 0; k < 4 && ok; ++k) {
          const MkGemm m = mk_gemm(a, l, k);
          const int u1 = m.p.start(c + 1);
          for (int u = m.p.start(c); u < u1; ++u) {
            if (wrap > 0 && !mbar_wait(&empty[st], (wrap & 1) ^ 1, flags)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[st], kWBlk);
            bulk_load_hint(ring + (size_t)st * a.stage_bytes, m.W + (size_t)u * kWBlk, kWBlk, &full[st], pol);
            if (++st == S) {
              st = 0;
              ++wrap;
            }
          }
        }
      if (!ok) raise_error(flags, a.err);
    }
  } else if (warp == 7) {
    if (lane == 0) {
      // ---------------------------------------------------------------- operand producer
      const uint32_t plane = (uint32_t)a.nt * 128;
      int st = 0, wrap = 0;
      bool ok = true;
      for (int l = 0; l < g.L && ok; ++l)
        for (int k = 0; k < 4 && ok; ++k) {
          const MkGemm m = mk_gemm(a, l, k);
          const CUtensorMap* xm = k == 1 ? &tmXo : (k == 3 ? &tmXa : &tmXh);
          const int u0 = m.p.start(c), u1 = m.p.start(c + 1);
          // whole-operand dependencies are awaited once per projection
          if (u0 < u1 && k != 3) {
            const unsigned* cnt = k == 0 ? mk_cnt(a, l, a.c.x_h) : (k == 1 ? mk_cnt(a, l, a.c.comb) : mk_cnt(a, l, a.c.x2));
            const unsigned target = k == 1 ? (unsigned)(n_tok * g.Hq) : (unsigned)n_tok;
            if (!counter_wait(cnt, target, flags, a.err)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();
            mk_mark(a, l, k == 0 ? 0 : (k == 1 ? 1 : 2), c0);
          }
          for (int u = u0; u < u1; ++u) {
            if (wrap > 0 && !mbar_wait(&empty[st], (wrap & 1) ^ 1, flags)) {
              ok = false;
              break;
            }
            const int kb = u % m.p.kb;
            if (k == 3) {   // down: the activation block of this K-range
              if (!counter_wait(mk_cnt(a, l, a.c.act) + kb, 1u, flags, a.err)) {
                ok = false;
                break;
              }
              fence_proxy_async_global();
              if (u == u0) mk_mark(a, l, 3, c0);
            }
            uint8_t* sx = ring + (size_t)st * a.stage_bytes + kWBlk;
            mbar_arrive_expect_tx(&full[st], 2 * plane);
            for (int r = 0; r < a.nt; r += 16) {
              tma_load_2d(sx + r * 128, xm, &full[st], kb * kTileK, r);
              tma_load_2d(sx + plane + r * 128, xm, &full[st], kb * kTileK, a.x_lo_row + r);
            }
            if (++st == S) {
              st = 0;
              ++wrap;
            }
          }
        }
      if (!ok) raise_error(flags, a.err);
    }
  } else if (warp == 6) {
    if (lane == 0 && has_item) {
      // ---------------------------------------------------------------- attention loader
      const int slot = a.rd->seq_slot[it_s];
      const int len = a.rd->len[it_s];
      int gp = 0;   // pages loaded so far (all layers)
      bool ok = true;
      auto load_page = [&](int l, int j) -> bool {
        const int st = gp & 1, use = gp >> 1;
        if (use > 0 && !mbar_wait(&kvempty[st], (use & 1) ^ 1, flags)) return false;
        const int page = a.btab[(long)slot * g.pages_per_seq + it_k0 / kPage + j];
        if (page < 0 || page >= g.max_pages) {
          atomicExch(a.err, DERR_BAD_PAGE);
          return false;
        }
        const long base = ((long)l * g.max_pages + page) * g.Hkv + it_kvh;
        uint8_t* sk = sKV + st * a.kv_stage_bytes;
        mbar_arrive_expect_tx(&kvfull[st], (uint32_t)a.kv_stage_bytes);
        for (int at = 0; at < a.datoms; ++at)
          tma_load_2d(sk + at * kKAtom, &tmK, &kvfull[st], at * 64, (int)(base * kPage));
        tma_load_2d(sk + a.datoms * kKAtom, &tmV, &kvfull[st], 0, (int)(base * g.d));
        ++gp;
        return true;
      };
      for (int l = 0; l < g.L && ok; ++l) {
        int j = 0;
        // context-only pages first: they were written before this round
        for (; ok && j < it_pages && j < kMkKvStages && it_k0 + (j + 1) * kPage <= len; ++j) ok = load_page(l, j);
        if (!ok) break;
        if (!counter_wait(mk_cnt(a, l, a.c.head) + it_kvh, (unsigned)(n_tok * (g.G + 2)), flags, a.err)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();
        if (l > 0 && !mbar_wait(qempty, (l - 1) & 1, flags)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(qfull, (uint32_t)(a.datoms * R * 128));
        for (int at = 0; at < a.datoms; ++at)
          tma_load_3d(sQ + at * kQAtom, &tmQ, qfull, at * 64, it_kvh * g.G, it_s * kBlock);
        for (; ok && j < it_pages; ++j) ok = load_page(l, j);
      }
      if (!ok) raise_error(flags, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint64_t d0 = desc_sw128(smem_u32(ring));
      const uint32_t dstage = (uint32_t)a.stage_bytes >> 4;
      constexpr uint32_t xo = kWBlk >> 4;
      const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
      int st = 0, wrap = 0, sg = 0;
      int gp = 0, gs = 0;   // attention pages and S tiles issued (all layers)
      bool ok = true;
      auto issue_s = [&](int j) -> bool {
        const int kst = (gp + j) & 1, kuse = (gp + j) >> 1;
        if (!mbar_wait(&kvfull[kst], kuse & 1, flags)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sKV + kst * a.kv_stage_bytes);
        const int sb = (gs + j) & 1;
        const uint32_t d_s = tatt + 128u + (uint32_t)(sb * 64);
        for (int kk = 0; kk < 4 * a.datoms; ++kk) {
          const int at = kk >> 2;
          const uint64_t adv = (uint64_t)((kk & 3) * 32) >> 4;
          mma_bf16(d_s, desc_sw128(q_addr + at * kQAtom) + adv, desc_sw128(k_addr + at * kKAtom) + adv, a.idesc_s,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(&sfull[sb]);
        return true;
      };
      for (int l = 0; l < g.L && ok; ++l)
        for (int k = 0; k < 4 && ok; ++k) {
          if (k == 1 && has_item) {
            // attention item of layer l
            if (!mbar_wait(qfull, l & 1, flags)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mk_mark(a, l, 4, c0);
            const int n = it_pages;
            if (n > 0) ok = issue_s(0);
            if (ok && n > 1) ok = issue_s(1);
            for (int j = 0; j < n && ok; ++j) {
              if (!mbar_wait(pfull, (gp + j) & 1, flags)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const int kst = (gp + j) & 1;
              const uint32_t v_addr = smem_u32(sKV + kst * a.kv_stage_bytes) + (uint32_t)(a.datoms * kKAtom);
#pragma unroll
              for (int kk = 0; kk < kPage / 16; ++kk) {
                const uint64_t adv = (uint64_t)(kk * 32) >> 4;
                mma_bf16(tatt, desc_sw128(p_addr) + adv, desc_sw128(v_addr) + adv, a.idesc_o,
                         (j > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(pvdone);
              mma_commit(&kvempty[kst]);
              if (j + 2 < n) ok = issue_s(j + 2);
            }
            mma_commit(qempty);   // every S MMA of this item has been issued
            mk_mark(a, l, 5, c0);
            gp += n;
            gs += n;
            if (!ok) break;
          }
          const MkGemm m = mk_gemm(a, l, k);
          const int u1 = m.p.start(c + 1);
          for (int u = m.p.start(c); u < u1 && ok; ++sg) {
            const int T = u / m.p.kb;
            const int seg_end = min(u1, (T + 1) * m.p.kb);
            const int b = sg & 1, use = sg >> 1;
            if (!mbar_wait(&accempty[b], (use & 1) ^ 1, flags)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(b * a.aw);
            for (int kk0 = 0; u < seg_end; ++u, ++kk0) {
              if (!mbar_wait(&full[st], wrap & 1, flags)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t dw = d0 + (uint64_t)(st * dstage);
              mma_bf16(d_tmem, dw, dw + xo, a.idesc_g, kk0 > 0 ? 1u : 0u);
#pragma unroll
              for (uint32_t kk = 2; kk < 8; kk += 2) mma_bf16(d_tmem, dw + kk, dw + xo + kk, a.idesc_g, 1u);
              mma_commit(&empty[st]);
              if (++st == S) {
                st = 0;
                ++wrap;
              }
            }
            if (ok) mma_commit(&accfull[b]);
          }
        }
      if (!ok) raise_error(flags, a.err);
      // every MMA this thread issued has completed before TMEM is released
      // (waited for even after an abort, within the time limit)
      mma_commit(fin);
      volatile int no_abort = 0;
      mbar_wait(fin, 0, &no_abort);
    }
  } else {
    // ------------------------------------------------------------------ compute warps
    const int ct = threadIdx.x - 64;        // 0..127
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int cw = warp - 2;                // compute warp 0..3
    int sg = 0;                             // projection segments drained (all layers)
    int pp = 0, gs = 0;                     // attention pages / S tiles consumed
    float4 v[kMkRowVec], w[kMkRowVec];

    auto prep_rows = [&](int l, const float* gain, bool second) {
      // norm(h) of row c into the operand planes of the next projection
      if (c >= n_tok) return;
      if (l > 0 || second) {
        const unsigned* dep = second ? mk_cnt(a, l, a.c.o_done) : mk_cnt(a, l - 1, a.c.down_done);
        group_wait(dep, (unsigned)grid, flags, a.err);
      }
      mk_row_norm(a.h + (size_t)c * g.H, gain, g.H, g.eps, v, w, red, ct);
      if (!flags[0]) {
#pragma unroll
        for (int k = 0; k < kMkRowVec; ++k) {
          const int i = ct + k * kMkCompute;
          if (4 * i < g.H) {
            const long idx = (long)c * g.H + 4 * i;
            put_operand(a.op_h, idx + 0, a.plane_h, v[k].x, 0);
            put_operand(a.op_h, idx + 1, a.plane_h, v[k].y, 0);
            put_operand(a.op_h, idx + 2, a.plane_h, v[k].z, 0);
            put_operand(a.op_h, idx + 3, a.plane_h, v[k].w, 0);
          }
        }
      }
      group_signal(mk_cnt(a, l, second ? a.c.x2 : a.c.x_h), flags);
    };

    // drain projection k of layer l; QKV and gate/up signal per tile, O and
    // down once per CTA
    auto drain = [&](int l, int k) {
      const MkGemm m = mk_gemm(a, l, k);
      const int u1 = m.p.start(c + 1);
      const int row = 32 * q + lane;
      for (int u = m.p.start(c); u < u1; ++sg) {
        const int T = u / m.p.kb;
        const int seg_end = min(u1, (T + 1) * m.p.kb);
        const int b = sg & 1, use = sg >> 1;
        const bool got = __all_sync(0xffffffffu, mbar_wait(&accfull[b], use & 1, flags));
        if (!got) raise_error(flags, a.err);
        __syncwarp();
        tc_fence_after();
        if (got) {
          float* dcol = m.dst + T * kTileN + row;
          const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * a.aw);
          for (int j0 = 0; j0 < n_tok; j0 += 16) {
            float x[16], y[16];
            tmem_ld16(base + (uint32_t)j0, x);
            tmem_ld16(base + (uint32_t)(a.nt + j0), y);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j0 + j < n_tok)
                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dcol + (long)(j0 + j) * m.dst_ld), "f"(x[j] + y[j])
                             : "memory");
          }
        }
        tc_fence_before();
        mbar_arrive(&accempty[b]);
        if (k == 0 || k == 2) group_signal(mk_cnt(a, l, k == 0 ? a.c.qkv_t : a.c.gu_t) + T, flags);
        u = seg_end;
      }
      if (k == 1 || k == 3) group_signal(mk_cnt(a, l, k == 1 ? a.c.o_done : a.c.down_done), flags);
    };

    // q/k head RMSNorm + RoPE of one (token, head) row of the QKV sums, by
    // one warp: q to the query buffer, k and v into the KV pages (block rows)
    auto qk_row = [&](int l, int tok, int hh) {
      const int d = g.d, half = d / 2, per = d / 32, dim0 = lane * per;
      const int kind = hh < g.Hq ? 0 : (hh < g.Hq + g.Hkv ? 1 : 2);
      const int head = kind == 0 ? hh : (kind == 1 ? hh - g.Hq : hh - g.Hq - g.Hkv);
      float* src = a.qkv_acc + (long)tok * g.qkv_n + hh * d + dim0;
      float x[4], gn[4];
      float2 cs[4];
      if (per == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
        x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
        *reinterpret_cast<float4*>(src) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
        x[0] = t.x, x[1] = t.y, x[2] = 0.f, x[3] = 0.f;
        *reinterpret_cast<float2*>(src) = make_float2(0.f, 0.f);
      }
      const float* gsrc = (kind == 0 ? a.qn : a.kn) + (size_t)l * d;
      for (int e = 0; e < per; ++e) {
        gn[e] = kind != 2 ? gsrc[dim0 + e] : 1.f;
        cs[e] = kind != 2 ? a.rope_cs[(long)tok * half + (dim0 + e) % half] : make_float2(1.f, 0.f);
      }
      if (kind != 2) {
        float ss = 0.f;
        for (int e = 0; e < per; ++e) ss += x[e] * x[e];
        ss = warp_sum(ss);
        const float rn = rsqrtf(ss / (float)d + g.eps);
        for (int e = 0; e < per; ++e) {
          const float y = x[e] * rn * gn[e];
          const float partner = __shfl_xor_sync(0xffffffffu, y, 16);   // dims j <-> j + d/2
          x[e] = lane < 16 ? (y * cs[e].x - partner * cs[e].y) : (y * cs[e].x + partner * cs[e].y);
        }
      }
      if (kind == 0) {
        const long qb = ((long)tok * g.Hq + head) * d + dim0;
        for (int e = 0; e < per; ++e) put_kv(a.q, qb + e, x[e], g.kvtype);
      } else {
        const int dst = a.rd->dest[tok];
        const int page = dst >> 6, off = dst & (kPage - 1);
        for (int e = 0; e < per; ++e) {
          if (kind == 1) put_kv(a.kpool, k_index(g, l, page, head, off, dim0 + e), x[e], g.kvtype);
          else put_kv(a.vpool, v_index(g, l, page, head, off, dim0 + e), x[e], g.kvtype);
        }
      }
      return kind == 0 ? head / g.G : head;
    };

    for (int l = 0; l < g.L; ++l) {
      prep_rows(l, a.in_ln + (size_t)l * g.H, false);
      drain(l, 0);
      if (ct == 0) mk_mark(a, l, 6, c0);

      // ---- q/k finish: rows c + grid*(cw + 4i), one warp per row
      {
        const int heads = g.Hq + 2 * g.Hkv;
        const int n_rows = n_tok * heads;
        for (int i = 0;; ++i) {
          const int r = c + grid * (cw + 4 * i);
          if (c + grid * 4 * i >= n_rows) break;   // CTA-uniform loop end
          if (r < n_rows) {
            const int tok = r / heads, hh = r % heads;
            const int T = hh * g.d / kTileN;
            bool ok = true;
            if (lane == 0) ok = counter_wait(mk_cnt(a, l, a.c.qkv_t) + T, contributors(a.pq, T), flags, a.err);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
              raise_error(flags, a.err);
            } else {
              const int grp = qk_row(l, tok, hh);
              fence_proxy_async_global();
              __syncwarp();
              if (lane == 0) counter_add(mk_cnt(a, l, a.c.head) + grp, 1);
            }
          }
        }
      }

      if (ct == 0) mk_mark(a, l, 7, c0);
      // ---- softmax of this CTA's attention item
      if (has_item) {
        const int r = 32 * q + lane;                  // query row of this thread
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int n = it_pages;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = !flags[0];
        for (int j = 0; j < n && ok; ++j) {
          const int sb = (gs + j) & 1, suse = (gs + j) >> 1;
          if (!__all_sync(0xffffffffu, mbar_wait(&sfull[sb], suse & 1, flags))) {
            ok = false;
            break;
          }
          __syncwarp();
          tc_fence_after();
          float sc[kPage];
          tmem_ld32(tatt + lane_base + 128u + (uint32_t)(sb * 64), sc);
          tmem_ld32(tatt + lane_base + 128u + (uint32_t)(sb * 64) + 32u, sc + 32);
          const int kc = min(kPage, it_k1 - (it_k0 + j * kPage));
          float mj = -INFINITY;
#pragma unroll
          for (int i = 0; i < kPage; ++i) {
            sc[i] = (i < kc) ? sc[i] * a.scale_log2 : -INFINITY;
            mj = fmaxf(mj, sc[i]);
          }
          const bool need = mj > m_run + kRescaleLog2;
          if (j > 0) {   // the single P buffer and O are free once P V^T of page j-1 is done
            if (!__all_sync(0xffffffffu, mbar_wait(pvdone, (pp + j - 1) & 1, flags))) {
              ok = false;
              break;
            }
            __syncwarp();
            tc_fence_after();
          }
          if (__any_sync(0xffffffffu, need && j > 0)) {
            const float alpha = need ? exp2f(m_run - mj) : 1.f;
            for (int cc = 0; cc < g.d / 32; ++cc) {
              float o[32];
              tmem_ld32(tatt + lane_base + (uint32_t)(cc * 32), o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(tatt + lane_base + (uint32_t)(cc * 32), o);
            }
            l_run *= alpha;
          }
          if (need) m_run = mj;
          float lsum = 0.f;
          uint8_t* prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t wv[4];
#pragma unroll
            for (int hq = 0; hq < 4; ++hq) {
              const float p0 = exp2f(sc[8 * cc + 2 * hq] - m_run);
              const float p1 = exp2f(sc[8 * cc + 2 * hq + 1] - m_run);
              lsum += p0 + p1;
              const __nv_bfloat162 bb = __floats2bfloat162_rn(p0, p1);
              wv[hq] = *reinterpret_cast<const uint32_t*>(&bb);
            }
            *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
          l_run += lsum;
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(pfull);
        }
        if (ok && n > 0 && __all_sync(0xffffffffu, mbar_wait(pvdone, (pp + n - 1) & 1, flags))) {
          __syncwarp();
          tc_fence_after();
          const long prow = (long)c * R + r;
          for (int cc = 0; cc < g.d / 32; ++cc) {
            float o[32];
            tmem_ld32(tatt + lane_base + (uint32_t)(cc * 32), o);
            if (r < R) {
              float4* dst = reinterpret_cast<float4*>(a.part_o + prow * g.d + cc * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
          }
          if (r < R) {
            a.part_ml[prow * 2] = m_run;
            a.part_ml[prow * 2 + 1] = l_run;
          }
        } else if (n > 0) {
          raise_error(flags, a.err);
        }
        tc_fence_before();
        pp += n;
        gs += n;
        group_signal(mk_cnt(a, l, a.c.att) + it_s * g.Hkv + it_kvh, flags);
        if (ct == 0) mk_mark(a, l, 8, c0);
      }

      // ---- split combine: (token, q head) rows, one warp per row (rows
      // c + grid*(cw + 4i)); lane owns d/32 dims, splits walked four deep
      {
        const int n_rows = n_tok * g.Hq;
        const int per = g.d / 32;
        const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
        for (int i = 0;; ++i) {
          if (c + grid * 4 * i >= n_rows) break;   // CTA-uniform loop end
          const int rr = c + grid * (cw + 4 * i);
          if (rr >= n_rows) continue;
          const int tok = rr / g.Hq, hq = rr % g.Hq;
          const int s = tok / kBlock, i16 = tok % kBlock;
          const int kvh = hq / g.G, r = i16 * g.G + hq % g.G;
          const int nsplit = (a.rd->item0[s + 1] - a.rd->item0[s]) / g.Hkv;
          const int it0 = a.rd->item0[s] + kvh * nsplit;
          bool ok = true;
          if (lane == 0) ok = counter_wait(mk_cnt(a, l, a.c.att) + s * g.Hkv + kvh, (unsigned)nsplit, flags, a.err);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            raise_error(flags, a.err);
            continue;
          }
          float M = -INFINITY;
          for (int sp = lane; sp < nsplit; sp += 32) M = fmaxf(M, __ldcg(ml + (long)(it0 + sp) * R + r).x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          float den = 0.f;
          for (int sp0 = 0; sp0 < nsplit; sp0 += 4) {
            float o[4][4];
            float2 mm[4];
#pragma unroll
            for (int kx = 0; kx < 4; ++kx) {
              const int sp = sp0 + kx;
              const long pr = (long)(it0 + sp) * R + r;
              mm[kx] = sp < nsplit ? __ldcg(ml + pr) : make_float2(-INFINITY, 0.f);
              if (per == 4) {
                const float4 t = sp < nsplit ? __ldcg(reinterpret_cast<const float4*>(a.part_o + pr * g.d) + lane)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                o[kx][0] = t.x, o[kx][1] = t.y, o[kx][2] = t.z, o[kx][3] = t.w;
              } else {
                const float2 t = sp < nsplit ? __ldcg(reinterpret_cast<const float2*>(a.part_o + pr * g.d) + lane)
                                             : make_float2(0.f, 0.f);
                o[kx][0] = t.x, o[kx][1] = t.y, o[kx][2] = 0.f, o[kx][3] = 0.f;
              }
            }
#pragma unroll
            for (int kx = 0; kx < 4; ++kx) {
              const float wgt = exp2f(mm[kx].x - M);
              den += wgt * mm[kx].y;
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[e] += wgt * o[kx][e];
            }
          }
          const float inv = 1.f / den;
          const long idx = (long)tok * (g.Hq * g.d) + hq * g.d + per * lane;
          for (int e = 0; e < per; ++e) put_operand(a.op_o, idx + e, a.plane_o, acc[e] * inv, 0);
          fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) counter_add(mk_cnt(a, l, a.c.comb), 1);
        }
      }

      if (ct == 0) mk_mark(a, l, 9, c0);
      drain(l, 1);
      if (ct == 0) mk_mark(a, l, 10, c0);
      prep_rows(l, a.post_ln + (size_t)l * g.H, true);
      if (ct == 0) mk_mark(a, l, 11, c0);
      drain(l, 2);
      if (ct == 0) mk_mark(a, l, 12, c0);

      // ---- SwiGLU of gate/up tiles c + grid*i (64 activation columns each)
      {
        const int n_tiles = a.pg.units / a.pg.kb;
        for (int T = c; T < n_tiles; T += grid) {
          group_wait(mk_cnt(a, l, a.c.gu_t) + T, contributors(a.pg, T), flags, a.err);
          if (!flags[0]) {
            for (int e = ct; e < n_tok * 64; e += kMkCompute) {
              const int tok = e >> 6, jj = e & 63;
              float* gp = a.gu_acc + (long)tok * 2 * g.I + T * kTileN + jj;
              const float gv = __ldcg(gp), uv = __ldcg(gp + 64);
              gp[0] = 0.f;
              gp[64] = 0.f;
              put_operand(a.op_a, (long)tok * g.I + T * 64 + jj, a.plane_a, gv / (1.f + __expf(-gv)) * uv, 0);
            }
          }
          group_signal(mk_cnt(a, l, a.c.act) + T, flags);
        }
      }

      drain(l, 3);
      if (ct == 0) mk_mark(a, l, 13, c0);
    }

    // ---- final norm of row c into the output
    if (c < n_tok) {
      group_wait(mk_cnt(a, g.L - 1, a.c.down_done), (unsigned)grid, flags, a.err);
      mk_row_norm(a.h + (size_t)c * g.H, a.fn, g.H, g.eps, v, w, red, ct);
      if (!flags[0]) {
        float4* o4 = reinterpret_cast<float4*>(a.out + (size_t)c * g.H);
#pragma unroll
        for (int k = 0; k < kMkRowVec; ++k) {
          const int i = ct + k * kMkCompute;
          if (4 * i < g.H) o4[i] = v[k];
        }
      }
    }
  }
  __syncwarp();   // role lanes rejoin their warp before the CTA barrier
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t round_mk_smem_bytes(int nt, int stages, int d) {
  const int datoms = d / 64;
  const int stage_bytes = kWBlk + 2 * nt * 128;
  const int kv_stage = datoms * kKAtom + d * 128;
  return (size_t)stages * stage_bytes + (size_t)datoms * kQAtom + kPBytes + (size_t)kMkKvStages * kv_stage + 512 +
         kMkCompute * 16 + 1024;
}

int round_mk_stages(int nt, int d) {
  const size_t fixed = round_mk_smem_bytes(nt, 0, d);
  const int stage_bytes = kWBlk + 2 * nt * 128;
  const long room = 227L * 1024 - (long)fixed;
  return (int)std::min<long>(12, room / stage_bytes);
}

cudaError_t launch_round_mk(const MkArgs& a0, int grid, const void* tmxh, const void* tmxo, const void* tmxa,
                            const void* tmq, const void* tmk, const void* tmv, cudaStream_t s) {
  MkArgs a = a0;
  a.idesc_g = idesc_bf16(kTileN, a.aw);
  a.idesc_s = idesc_bf16(128, kPage);
  a.idesc_o = idesc_bf16(128, a.g.d);
  const size_t smem = round_mk_smem_bytes(a.nt, a.stages, a.g.d);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(round_mk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_bytes = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, round_mk_kernel, *static_cast<const CUtensorMap*>(tmxh),
                            *static_cast<const CUtensorMap*>(tmxo), *static_cast<const CUtensorMap*>(tmxa),
                            *static_cast<const CUtensorMap*>(tmq), *static_cast<const CUtensorMap*>(tmk),
                            *static_cast<const CUtensorMap*>(tmv), a);
}

}  // namespace dfl
