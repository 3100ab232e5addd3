// attn_tc.cu -- non-causal block attention over the paged KV cache on the
// 5th-generation tensor cores.
//
// One CTA per work item (sequence, kv head, split of the keys [cached context
// ; 16 block rows]).  The G q-heads x 16 block rows that share a kv head form
// one M = 128 query tile (rows padded with zeros when G*16 < 128), so each
// K/V page is read once per item:
//   warp 0 (one lane)  TMA: the query tile, then the split's K pages [64 x d]
//                      and V^T pages [d x 64] through a ring of stages;
//   warp 1 (one lane)  tcgen05.mma: S = Q K^T into one of two TMEM buffers,
//                      then O += P V^T into the TMEM output accumulator;
//   warps 2..5         softmax, one thread per query row: scores from TMEM,
//                      exp2 with a running max, P (bf16) into one of two
//                      shared-memory buffers in the 128-byte swizzle the MMA
//                      reads, so page j+1's softmax overlaps page j's P V^T.  O is rescaled only
//                      when a row's max grows by more than 2^8 (exact: the
//                      final division uses the same max).
// Each item writes its unnormalised O with (max, sum); the combine kernel
// merges the splits (all in log2 units).
#include <algorithm>
#include <cmath>

#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

struct AttnTcCfg {
  int datoms;        // d / 64 (K-atoms of a row)
  int stages;
  int stage_bytes;   // K page (datoms x 8 KB) + V^T page (d x 128 B)
  uint32_t idesc_s;  // M=128, N=64
  uint32_t idesc_o;  // M=128, N=d
  float scale_log2;  // log2(e) / sqrt(d)
};

constexpr int kAttnThreads = 192;
constexpr int kQAtomBytes = 128 * 128;   // 128 rows x 128 B
constexpr int kKAtomBytes = 64 * 128;    // 64 keys x 128 B
constexpr float kRescaleLog2 = 8.f;

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, AttnArgs a, AttnTcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geo& g = a.g;
  uint8_t* sQ = smem;                                   // datoms x 16 KB
  uint8_t* sP = sQ + t.datoms * kQAtomBytes;            // 2 x 16 KB (P of pages j, j+1)
  uint8_t* sKV = sP + 2 * kQAtomBytes;                  // stages x stage_bytes
  uint8_t* ctl = sKV + t.stages * t.stage_bytes;
  uint64_t* kvfull = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* kvempty = kvfull + t.stages;
  uint64_t* sfull = kvempty + t.stages;                 // [2]
  uint64_t* qfull = sfull + 2;
  uint64_t* pfull = qfull + 1;                          // [2]
  uint64_t* pvdone = pfull + 2;                         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pvdone + 2);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long c0 = 0;
  if (threadIdx.x == 0) trace_entry(a.trace, blockIdx.x, &c0);
  if (a.trace) {
    __shared__ unsigned long long c0_shared;
    if (threadIdx.x == 0) c0_shared = c0;
    __syncthreads();
    c0 = c0_shared;
  }
  const int R = g.G * kBlock;
  // zero the query tile's padding rows (the MMA reads all 128 rows)
  for (int idx = threadIdx.x; idx < t.datoms * (128 - R) * 32; idx += kAttnThreads) {
    const int atom = idx / ((128 - R) * 32), rem = idx % ((128 - R) * 32);
    reinterpret_cast<uint32_t*>(sQ + atom * kQAtomBytes + R * 128)[rem] = 0u;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(qfull, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], kEpiThreads);
      mbar_init(&pvdone[b], 1);
    }
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 1, c0);  // 1: set-up done

  // The descriptor, the page table and the cached-context pages were written
  // by kernels that completed before the predecessor passed its own launch
  // wait (which is when this kernel may start), so they are read before this
  // kernel's wait; only the pages holding this round's block rows and the
  // query tile (both written by the predecessor) wait for it.
  const int item = blockIdx.x;
  int s, kvh, k0, k1;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1);
  const int n_pages = (k1 - k0 + kPage - 1) / kPage;
  const int n_all = n_pages;
  const int slot = a.rd->seq_slot[s];
  const int len = a.rd->len[s];

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      auto load_page = [&](int j) -> bool {
        const int st = j % t.stages;
        const int page = a.block_table[(long)slot * g.pages_per_seq + k0 / kPage + j];
        if (page < 0 || page >= g.max_pages) {
          atomicExch(a.err, DERR_BAD_PAGE);
          return false;
        }
        const long base = ((long)a.layer * g.max_pages + page) * g.Hkv + kvh;
        uint8_t* st_k = sKV + st * t.stage_bytes;
        uint8_t* st_v = st_k + t.datoms * kKAtomBytes;
        mbar_arrive_expect_tx(&kvfull[st], (uint32_t)t.stage_bytes);
        for (int at = 0; at < t.datoms; ++at)
          tma_load_2d(st_k + at * kKAtomBytes, &tmK, &kvfull[st], at * 64, (int)(base * kPage));
        tma_load_2d(st_v, &tmV, &kvfull[st], 0, (int)(base * g.d));
        return true;
      };
      bool ok = true;
      int j = 0;
      // context-only pages that fit the ring, before the launch wait
      for (; ok && j < n_pages && j < t.stages && k0 + (j + 1) * kPage <= len; ++j) ok = load_page(j);
      pdl_wait();
      pdl_launch_dependents();
      mbar_arrive_expect_tx(qfull, (uint32_t)(t.datoms * R * 128));
      for (int at = 0; at < t.datoms; ++at)
        tma_load_3d(sQ + at * kQAtomBytes, &tmQ, qfull, at * 64, kvh * g.G, s * kBlock);
      for (; ok && j < n_pages; ++j) {
        const int st = j % t.stages;
        if (j >= t.stages && !mbar_wait(&kvempty[st], ((j / t.stages) & 1) ^ 1, &flags[0])) {
          ok = false;
          break;
        }
        ok = load_page(j);
      }
      if (!ok) flags[0] = 1;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(qfull, 0, &flags[0]);
      tc_fence_after();
      trace_mark(a.trace, blockIdx.x, 2, c0);                   // 2: query tile ready
      const uint32_t q_addr = smem_u32(sQ);
      auto kv_addr = [&](int j) -> uint32_t { return smem_u32(sKV + (j % t.stages) * t.stage_bytes); };
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait(&kvfull[j % t.stages], (j / t.stages) & 1, &flags[0])) return false;
        tc_fence_after();
        const uint32_t k_addr = kv_addr(j);
        const uint32_t d_s = tmem + 128u + (uint32_t)((j & 1) * 64);
        for (int kk = 0; kk < 4 * t.datoms; ++kk) {
          const int at = kk >> 2;
          const uint64_t adv = (uint64_t)((kk & 3) * 32) >> 4;
          mma_bf16(d_s, desc_sw128(q_addr + at * kQAtomBytes) + adv, desc_sw128(k_addr + at * kKAtomBytes) + adv,
                   t.idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sfull[j & 1]);
        return true;
      };
      if (ok && n_all > 0) ok = issue_s(0);
      if (ok && n_all > 1) ok = issue_s(1);
      for (int j = 0; j < n_all && ok; ++j) {
        if (!mbar_wait(&pfull[j & 1], (j >> 1) & 1, &flags[0])) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t p_addr = smem_u32(sP + (j & 1) * kQAtomBytes);
        const uint32_t v_addr = kv_addr(j) + (uint32_t)(t.datoms * kKAtomBytes);
#pragma unroll
        for (int kk = 0; kk < kPage / 16; ++kk) {
          const uint64_t adv = (uint64_t)(kk * 32) >> 4;
          mma_bf16(tmem, desc_sw128(p_addr) + adv, desc_sw128(v_addr) + adv, t.idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pvdone[j & 1]);
        mma_commit(&kvempty[j % t.stages]);
        if (j + 2 < n_all) ok = issue_s(j + 2);
      }
      if (!ok) flags[0] = 1;
      trace_mark(a.trace, blockIdx.x, 3, c0);                   // 3: last MMA issued
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    pdl_wait();
    const int q = warp & 3;
    const int r = 32 * q + lane;                 // query row of this thread
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_all; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sfull[j & 1], (j >> 1) & 1, &flags[0]))) {
        ok = false;
        break;
      }
      __syncwarp();
      tc_fence_after();
      float sc[kPage];
      tmem_ld32(tmem + lane_base + 128u + (uint32_t)((j & 1) * 64), sc);
      tmem_ld32(tmem + lane_base + 128u + (uint32_t)((j & 1) * 64) + 32u, sc + 32);
      const int kc = min(kPage, k1 - (k0 + j * kPage));
      float mj = -INFINITY;
#pragma unroll
      for (int i = 0; i < kPage; ++i) {
        sc[i] = (i < kc) ? sc[i] * t.scale_log2 : -INFINITY;
        mj = fmaxf(mj, sc[i]);
      }
      const bool need = mj > m_run + kRescaleLog2;
      // P buffer j&1 is free once O += P V^T of page j-2 has completed
      if (j >= 2) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pvdone[j & 1], ((j - 2) >> 1) & 1, &flags[0]))) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
      }
      const bool resc = __any_sync(0xffffffffu, need && j > 0);
      // rescaling O needs every product issued so far (through page j-1) done
      if (resc) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1, &flags[0]))) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
      }
      if (resc) {
        const float alpha = need ? exp2f(m_run - mj) : 1.f;
        for (int c = 0; c < g.d / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + (uint32_t)(c * 32), o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + lane_base + (uint32_t)(c * 32), o);
        }
        l_run *= alpha;
      }
      if (need) m_run = mj;
      float lsum = 0.f;
      uint8_t* prow = sP + (j & 1) * kQAtomBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float p0 = exp2f(sc[8 * c + 2 * h] - m_run);
          const float p1 = exp2f(sc[8 * c + 2 * h + 1] - m_run);
          lsum += p0 + p1;
          const __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);
          w[h] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&pfull[j & 1]);
    }
    if (ok && n_all > 0 &&
        __all_sync(0xffffffffu, mbar_wait(&pvdone[(n_all - 1) & 1], ((n_all - 1) >> 1) & 1, &flags[0]))) {
      __syncwarp();
      tc_fence_after();
      const long prow = (long)item * R + r;
      for (int c = 0; c < g.d / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_base + (uint32_t)(c * 32), o);
        if (r < R) {
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow * g.d + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      if (r < R) {
        a.part_ml[prow * 2] = m_run;
        a.part_ml[prow * 2 + 1] = l_run;
      }
    } else if (n_all > 0) {
      flags[0] = 1;
    }
  }
  if (threadIdx.x == 64) trace_mark(a.trace, blockIdx.x, 4, c0);   // 4: softmax warps done
  __syncwarp();   // role lanes rejoin their warp before the CTA barrier
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 5, c0);     // 5: exit
  if (threadIdx.x == 64) trace_mark(a.trace, blockIdx.x, 7, c0);
  if (flags[0] && threadIdx.x == 0) atomicExch(a.err, DERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

size_t attn_tc_smem_bytes(int d, int stages) {
  const int datoms = d / 64;
  const int stage_bytes = datoms * kKAtomBytes + d * 128;
  return (size_t)datoms * kQAtomBytes + 2 * kQAtomBytes + (size_t)stages * stage_bytes + 256 + 1024;
}

void launch_attention_tc(const AttnArgs& a, int n_items, const void* tmq, const void* tmk, const void* tmv,
                         cudaStream_t s) {
  AttnTcCfg t{};
  const int d = a.g.d;
  t.datoms = d / 64;
  t.stage_bytes = t.datoms * kKAtomBytes + d * 128;
  t.stages = 4;
  t.idesc_s = idesc_bf16(128, kPage);
  t.idesc_o = idesc_bf16(128, d);
  t.scale_log2 = 1.4426950408889634f / std::sqrt((float)d);
  const size_t smem = attn_tc_smem_bytes(d, t.stages);
  static size_t attr_bytes = 0;
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return;
    attr_bytes = smem;
  }
  launch_pdl(attn_tc_kernel, dim3(n_items), dim3(kAttnThreads), smem, s, *static_cast<const CUtensorMap*>(tmq),
             *static_cast<const CUtensorMap*>(tmk), *static_cast<const CUtensorMap*>(tmv), a, t);
}

}  // namespace dfl
