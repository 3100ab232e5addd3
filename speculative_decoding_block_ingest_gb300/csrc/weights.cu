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

// e4m3 weights stay one byte each: block (T, kb) of 128 rows x 64 codes is
// an 8 KB unit at index T * (K/64) + kb, row r at byte r * 64 with its 16-code
// piece p at piece position p ^ ((r >> 1) & 3), so that eight consecutive rows'
// pieces fall in eight different shared-memory bank groups when a thread per
// row reads them.  The projection widens the codes to f16 (exact) in shared
// memory; the per-row scales multiply the sums as the projection drains.
__global__ void repack_e4m3_kernel(uint8_t* dst, int K, const uint8_t* src, int n_rows, int chunk, int stride,
                                   int base) {
  const int ppr = K / 16;   // 16-code pieces per row
  const long n = (long)n_rows * ppr;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
    const int i = (int)(idx / ppr), c = (int)(idx % ppr);
    const int R = base + (i / chunk) * stride + i % chunk;
    const int T = R / kTileN, r = R % kTileN, kb = c / 4, p = c % 4;
    const size_t off = ((size_t)T * (K / kTileK) + kb) * (kTileN * kTileK) + (size_t)r * 64 + ((p ^ ((r >> 1) & 3)) * 16);
    *reinterpret_cast<uint4*>(dst + off) = *reinterpret_cast<const uint4*>(src + (size_t)i * K + (size_t)c * 16);
  }
}

void launch_repack_e4m3(void* dst, int K, const void* src, int n_rows, int chunk, int stride, int base,
                        cudaStream_t s) {
  const long n = (long)n_rows * (K / 16);
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
