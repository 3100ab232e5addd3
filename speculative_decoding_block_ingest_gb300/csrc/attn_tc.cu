// attn_tc.cu -- non-causal block attention over the paged KV cache on the
// 5th-generation tensor cores.
//
// One CTA per work item (sequence, kv head, split of the cached keys).  The
// G q-heads x 16 block rows that share a kv head form one M = 128 query tile
// (rows padded with zeros when G*16 < 128), so each K/V page is read once per
// item:
//   warp 0 (one lane)  TMA: the split's K pages [64 x d] and V^T pages
//                      [d x 64] through a ring of stages;
//   warp 1 (one lane)  tcgen05.mma: S = Q K^T into one of two TMEM buffers,
//                      then O += P V^T into the TMEM output accumulator;
//   warps 2..5         first build the query tile from the QKV accumulator
//                      (input-norm scale, q head RMSNorm, RoPE, bf16) and, in
//                      a sequence's last split, the 16 block rows' K and V^T
//                      as one more "page" in shared memory (the block's K/V are
//                      transient: they never go to HBM); then the softmax, one
//                      thread per query row: scores from TMEM, exp2 with a
//                      running max, P (bf16) into shared memory in the
//                      128-byte swizzle the MMA reads.  O is rescaled only when
//                      a row's max grows by more than 2^8 (exact: the final
//                      division uses the same max).
// The query tile is built while the first K/V pages stream in.  Each item
// writes its unnormalised O with (max, sum); the combine kernel merges the
// splits (all in log2 units).
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

// Byte offset of element (row, col) (col in bf16 units, < 64) in a K-major
// 128-byte-swizzled atom.
__device__ __forceinline__ int sw128_off(int row, int col) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2;
}

// Write lane's PER dims of one row into a K-major tile of atoms atom_bytes apart.
template <int PER>
__device__ __forceinline__ void put_row_bf16(uint8_t* tile, int atom_bytes, int row, const float* x) {
  const int lane = threadIdx.x & 31;
  const int dim0 = lane * PER;
  uint8_t* at = tile + (dim0 >> 6) * atom_bytes + sw128_off(row, dim0 & 63);
  if (PER == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    *reinterpret_cast<uint2*>(at) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    *reinterpret_cast<uint32_t*>(at) = *reinterpret_cast<const uint32_t*>(&a);
  }
}

// Rows of the QKV accumulator for the query tile (block == false: rows
// r = token * G + local head) or the block page (block == true: the 16 block
// rows' K, normed and roped, and V^T).  Each builder warp handles 4 rows per
// step and issues all of their loads before any arithmetic.
template <int PER>
__device__ __forceinline__ void build_tiles(const AttnArgs& a, int s, int kvh, bool block, uint8_t* sQ, uint8_t* sBK,
                                            uint8_t* sBV) {
  const Geo& g = a.g;
  constexpr int d = 32 * PER, half = d / 2;
  const int warp = (threadIdx.x >> 5) - 2, lane = threadIdx.x & 31;
  const int dim0 = lane * PER;
  const int ld = g.qkv_n;
  const int rows = block ? kBlock : g.G * kBlock;
  const float* gsrc = block ? a.kn : a.qn;
  float gn[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) gn[q] = gsrc[dim0 + q];
  for (int r0 = warp * 4; r0 < rows; r0 += 16) {
    float x[4][PER], v[4][PER], rs[4];
    float2 cs[4][PER];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u;
      if (r >= rows) continue;
      const int i = block ? r : r / g.G;
      const int tok = s * kBlock + i;
      const int col0 = block ? (g.Hq + kvh) * d : (kvh * g.G + r % g.G) * d;
      const float* src = a.qkv + (long)tok * ld + col0 + dim0;
      if (PER == 4) {
        const float4 t4 = __ldcg(reinterpret_cast<const float4*>(src));
        x[u][0] = t4.x; x[u][1] = t4.y; x[u][2] = t4.z; x[u][3] = t4.w;
      } else {
        const float2 t2 = __ldcg(reinterpret_cast<const float2*>(src));
        x[u][0] = t2.x; x[u][1] = t2.y;
      }
      if (block) {
        const float* vsrc = a.qkv + (long)tok * ld + (g.Hq + g.Hkv + kvh) * d + dim0;
#pragma unroll
        for (int q = 0; q < PER; ++q) v[u][q] = __ldcg(vsrc + q);
      }
      rs[u] = a.r_in[tok];
#pragma unroll
      for (int q = 0; q < PER; ++q) cs[u][q] = a.rope_cs[(long)tok * half + (dim0 + q) % half];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u;
      if (r >= rows) continue;
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        x[u][q] *= rs[u];
        ss += x[u][q] * x[u][q];
      }
      ss = warp_sum(ss);
      const float rn = rsqrtf(ss / (float)d + g.eps);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const float y = x[u][q] * rn * gn[q];
        const float partner = __shfl_xor_sync(0xffffffffu, y, 16);   // dims j <-> j + d/2
        x[u][q] = lane < 16 ? (y * cs[u][q].x - partner * cs[u][q].y) : (y * cs[u][q].x + partner * cs[u][q].y);
      }
      if (!block) {
        put_row_bf16<PER>(sQ, kQAtomBytes, r, x[u]);
      } else {
        put_row_bf16<PER>(sBK, kKAtomBytes, r, x[u]);
#pragma unroll
        for (int q = 0; q < PER; ++q)
          *reinterpret_cast<__nv_bfloat16*>(sBV + sw128_off(dim0 + q, r)) = __float2bfloat16_rn(v[u][q] * rs[u]);
      }
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs a,
                   AttnTcCfg t) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geo& g = a.g;
  uint8_t* sQ = smem;                                   // datoms x 16 KB
  uint8_t* sP = sQ + t.datoms * kQAtomBytes;            // 16 KB
  uint8_t* sB = sP + kQAtomBytes;                       // block "page": K then V^T (stage_bytes)
  uint8_t* sKV = sB + t.stage_bytes;                    // stages x stage_bytes
  uint8_t* ctl = sKV + t.stages * t.stage_bytes;
  uint64_t* kvfull = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* kvempty = kvfull + t.stages;
  uint64_t* sfull = kvempty + t.stages;                 // [2]
  uint64_t* qfull = sfull + 2;
  uint64_t* bfull = qfull + 1;
  uint64_t* pfull = bfull + 1;
  uint64_t* pvdone = pfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pvdone + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);   // abort
  uint8_t* sBV = sB + t.datoms * kKAtomBytes;

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
  // zero the query tile's padding rows and the whole block page (its unused
  // key rows / columns must read as zeros)
  for (int idx = threadIdx.x; idx < t.datoms * (128 - R) * 32; idx += kAttnThreads) {
    const int atom = idx / ((128 - R) * 32), rem = idx % ((128 - R) * 32);
    reinterpret_cast<uint32_t*>(sQ + atom * kQAtomBytes + R * 128)[rem] = 0u;
  }
  for (int idx = threadIdx.x; idx < t.stage_bytes / 16; idx += kAttnThreads)
    reinterpret_cast<uint4*>(sB)[idx] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < t.stages; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(qfull, kEpiThreads);
    mbar_init(bfull, kEpiThreads);
    mbar_init(pfull, kEpiThreads);
    mbar_init(pvdone, 1);
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x == 0) trace_mark(a.trace, blockIdx.x, 1, c0);  // 1: set-up and launch wait done

  const int item = blockIdx.x;
  int s, kvh, k0, k1;
  bool last;
  attn_item(a.rd, g.Hkv, item, &s, &kvh, &k0, &k1, &last);
  const int n_pages = (k1 - k0 + kPage - 1) / kPage;     // cached-key pages
  const int n_all = n_pages + (last ? 1 : 0);            // plus the block page
  const int slot = a.rd->seq_slot[s];

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      for (int j = 0; j < n_pages; ++j) {
        const int st = j % t.stages;
        if (j >= t.stages && !mbar_wait(&kvempty[st], ((j / t.stages) & 1) ^ 1, &flags[0])) {
          flags[0] = 1;
          break;
        }
        const int page = a.block_table[(long)slot * g.pages_per_seq + k0 / kPage + j];
        if (page < 0 || page >= g.max_pages) {
          atomicExch(a.err, DERR_BAD_PAGE);
          flags[0] = 1;
          break;
        }
        const long base = ((long)a.layer * g.max_pages + page) * g.Hkv + kvh;
        uint8_t* st_k = sKV + st * t.stage_bytes;
        uint8_t* st_v = st_k + t.datoms * kKAtomBytes;
        mbar_arrive_expect_tx(&kvfull[st], (uint32_t)t.stage_bytes);
        for (int at = 0; at < t.datoms; ++at)
          tma_load_2d(st_k + at * kKAtomBytes, &tmK, &kvfull[st], at * 64, (int)(base * kPage));
        tma_load_2d(st_v, &tmV, &kvfull[st], 0, (int)(base * g.d));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(qfull, 0, &flags[0]);
      tc_fence_after();
      trace_mark(a.trace, blockIdx.x, 2, c0);                   // 2: query tile ready
      const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
      auto kv_addr = [&](int j) -> uint32_t {
        return j < n_pages ? smem_u32(sKV + (j % t.stages) * t.stage_bytes) : smem_u32(sB);
      };
      auto issue_s = [&](int j) -> bool {
        if (j < n_pages) {
          if (!mbar_wait(&kvfull[j % t.stages], (j / t.stages) & 1, &flags[0])) return false;
        } else {
          if (!mbar_wait(bfull, 0, &flags[0])) return false;
        }
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
        if (!mbar_wait(pfull, j & 1, &flags[0])) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_addr = kv_addr(j) + (uint32_t)(t.datoms * kKAtomBytes);
#pragma unroll
        for (int kk = 0; kk < kPage / 16; ++kk) {
          const uint64_t adv = (uint64_t)(kk * 32) >> 4;
          mma_bf16(tmem, desc_sw128(p_addr) + adv, desc_sw128(v_addr) + adv, t.idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(pvdone);
        if (j < n_pages) mma_commit(&kvempty[j % t.stages]);
        if (j + 2 < n_all) ok = issue_s(j + 2);
      }
      if (!ok) flags[0] = 1;
      trace_mark(a.trace, blockIdx.x, 3, c0);                   // 3: last MMA issued
    }
  } else {
    // ------------------------------------------------------------------ tile builders, then softmax
    if (g.d == 128) build_tiles<4>(a, s, kvh, false, sQ, sB, sBV);
    else build_tiles<2>(a, s, kvh, false, sQ, sB, sBV);
    fence_proxy_async_smem();
    mbar_arrive(qfull);
    if (last) {
      if (g.d == 128) build_tiles<4>(a, s, kvh, true, sQ, sB, sBV);
      else build_tiles<2>(a, s, kvh, true, sQ, sB, sBV);
      fence_proxy_async_smem();
      mbar_arrive(bfull);
    }
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
      const int kc = j < n_pages ? min(kPage, k1 - (k0 + j * kPage)) : kBlock;
      float mj = -INFINITY;
#pragma unroll
      for (int i = 0; i < kPage; ++i) {
        sc[i] = (i < kc) ? sc[i] * t.scale_log2 : -INFINITY;
        mj = fmaxf(mj, sc[i]);
      }
      const bool need = mj > m_run + kRescaleLog2;
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(pvdone, (j - 1) & 1, &flags[0]))) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need && j > 0)) {
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
      uint8_t* prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
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
      mbar_arrive(pfull);
    }
    if (ok && n_all > 0 && __all_sync(0xffffffffu, mbar_wait(pvdone, (n_all - 1) & 1, &flags[0]))) {
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
  return (size_t)datoms * kQAtomBytes + kQAtomBytes + (size_t)(stages + 1) * stage_bytes + 256 + 1024;
}

void launch_attention_tc(const AttnArgs& a, int n_items, const void* tmk, const void* tmv, cudaStream_t s) {
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
  launch_pdl(attn_tc_kernel, dim3(n_items), dim3(kAttnThreads), smem, s, *static_cast<const CUtensorMap*>(tmk),
             *static_cast<const CUtensorMap*>(tmv), a, t);
}

}  // namespace dfl
