// static_full.cu -- the fixed device region behind dflash_forward_full_static.
//
// A file-scope device array holds the context K/V pages of one first-light
// forward, so that entry point needs no page of the handle's KV pool and
// allocates nothing.  It serves callers that cannot allocate: once every pool
// page belongs to a live sequence, the only way to more pages is a larger
// workspace, i.e. a new device allocation plus a copy of every live page.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.cuh"

namespace dfl {

// Zero when the library's device code is loaded.  Rows past a call's last
// key in its last page are read by the attention (and masked), so they must
// stay finite: zero or an earlier call's K/V in the same format.  Another
// handle's rows (another drafter, maybe another element format: bf16 or f32
// bytes read as e4m3 can be NaN codes) are not, so a handle's first call
// after another handle's clears the region.
static __device__ __align__(256) unsigned char g_fixed_kv[kFixedKvBytes];

// Device address of the region on the current device.  The first call on a
// device (with that device current) looks it up once.  *fresh: the region
// was last used by a handle other than `user` (the caller clears it); `user`
// is recorded as the last user (0, an id no handle has, marks it unclaimed).
cudaError_t fixed_kv_region(void** base, uint64_t user, bool* fresh) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kFixedMaxDevices) return cudaErrorInvalidDevice;
  static std::mutex mu;
  static void* addr[kFixedMaxDevices] = {};
  static uint64_t last_user[kFixedMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fixed_kv);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *base = addr[dev];
  *fresh = last_user[dev] != user;
  last_user[dev] = user;
  return cudaSuccess;
}

}  // namespace dfl
