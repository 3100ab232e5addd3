// weights.cu -- weight blocks for the tensor-core projections.
//
// A bf16 projection [N][K] is stored as (N/128) x (K/64) blocks of 16 KB;
// block (T, kb) holds rows 128T..128T+127 and columns 64kb..64kb+63 already in
// the shared-memory image the MMA reads: row r at byte r*128, its 16-byte
// chunk c at chunk position c ^ (r & 7) (the 128-byte swizzle).  Block
// (T, kb) sits at index T * (K/64) + kb, the projection's unit number, so a
// CTA's run of units is one contiguous HBM stream fetched by plain bulk copies
// of 16 KB.
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdint>

#include "kernels.cuh"

namespace dfl {

// Source rows i in [0, n_rows) land on logical rows
// base + (i / chunk) * stride + i % chunk (chunk = n_rows: contiguous).
__global__ void repack_kernel(uint8_t* dst, int K, const uint16_t* src, int n_rows, int chunk, int stride,
                              int base) {
  const int cpr = K / 8;   // 16-byte chunks per row
  const long n = (long)n_rows * cpr;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
    const int i = (int)(idx / cpr), c = (int)(idx % cpr);
    const int R = base + (i / chunk) * stride + i % chunk;
    const int T = R / kTileN, r = R % kTileN, kb = c / 8, c16 = c % 8;
    const size_t off = ((size_t)T * (K / kTileK) + kb) * (kTileN * kTileK * 2) + (size_t)r * 128 + ((c16 ^ (r & 7)) * 16);
    *reinterpret_cast<uint4*>(dst + off) = *reinterpret_cast<const uint4*>(src + (size_t)i * K + (size_t)c * 8);
  }
}

// The same blocks from OCP e4m3 bytes: every e4m3 value is exactly a bf16
// value, so the expansion is exact (the per-row scales are applied where the
// projections drain their accumulators).
__global__ void repack_e4m3_kernel(uint8_t* dst, int K, const uint8_t* src, int n_rows, int chunk, int stride,
                                   int base) {
  const int cpr = K / 8;   // 8-element chunks per row (16 bytes of bf16)
  const long n = (long)n_rows * cpr;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
    const int i = (int)(idx / cpr), c = (int)(idx % cpr);
    const int R = base + (i / chunk) * stride + i % chunk;
    const int T = R / kTileN, r = R % kTileN, kb = c / 8, c16 = c % 8;
    const size_t off = ((size_t)T * (K / kTileK) + kb) * (kTileN * kTileK * 2) + (size_t)r * 128 + ((c16 ^ (r & 7)) * 16);
    const uint2 raw = *reinterpret_cast<const uint2*>(src + (size_t)i * K + (size_t)c * 8);
    const uint8_t* b = reinterpret_cast<const uint8_t*>(&raw);
    __nv_bfloat16 out[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      __nv_fp8_e4m3 v;
      v.__x = b[e];
      out[e] = __float2bfloat16_rn(static_cast<float>(v));
    }
    *reinterpret_cast<uint4*>(dst + off) = *reinterpret_cast<const uint4*>(out);
  }
}

void launch_repack_e4m3(void* dst, int K, const void* src, int n_rows, int chunk, int stride, int base,
                        cudaStream_t s) {
  const long n = (long)n_rows * (K / 8);
  const int grid = (int)std::min<long>((n + 255) / 256, 8192);
  if (n > 0)
    repack_e4m3_kernel<<<grid, 256, 0, s>>>(static_cast<uint8_t*>(dst), K, static_cast<const uint8_t*>(src), n_rows,
                                             chunk, stride, base);
}

void launch_repack(void* dst, int K, const void* src, int n_rows, int chunk, int stride, int base, cudaStream_t s) {
  const long n = (long)n_rows * (K / 8);
  const int grid = (int)std::min<long>((n + 255) / 256, 8192);
  if (n > 0)
    repack_kernel<<<grid, 256, 0, s>>>(static_cast<uint8_t*>(dst), K, static_cast<const uint16_t*>(src), n_rows,
                                        chunk, stride, base);
}

}  // namespace dfl
