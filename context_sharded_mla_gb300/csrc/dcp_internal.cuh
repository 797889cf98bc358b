// dcp_internal.cuh — helpers shared by the library's translation units.
//
// Layout arithmetic of the sharded KV cache (block round-robin with interleave
// I; I = 1 is token round-robin).  Sources: "Decode Context Parallelism"
// (zdszero), "Core abstraction" idea 1; "PCP / DCP：计算、KV 布局与块轮转",
// section 6 (owner, local_index, local_len) and section "KV cache 管理"
// (slot = page_id * page_size + offset).
#pragma once

#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dcp.h"

namespace dcp {

constexpr int kDk = 576;   // latent row: 512 c_K + 64 k_R
constexpr int kDv = 512;   // value dims (c_K)

struct Layout {
  int64_t N, I, P;
};

__host__ __device__ inline int64_t owner_of(int64_t p, const Layout& L) { return (p / L.I) % L.N; }

__host__ __device__ inline int64_t local_row_of(int64_t p, const Layout& L) {
  return (p / (L.N * L.I)) * L.I + p % L.I;
}

// Positions in [0, x) owned by shard r.
__host__ __device__ inline int64_t count_of(int64_t r, int64_t x, const Layout& L) {
  const int64_t blk = L.N * L.I;
  int64_t rem = x % blk - r * L.I;
  rem = rem < 0 ? 0 : (rem > L.I ? L.I : rem);
  return (x / blk) * L.I + rem;
}

inline bool layout_ok(const dcp_layout_t* l) {
  return l && l->n_shards >= 1 && l->interleave >= 1 && l->page_size >= 1 &&
         l->page_size % l->interleave == 0;
}

inline Layout to_layout(const dcp_layout_t* l) {
  return Layout{l->n_shards, l->interleave, l->page_size};
}

__device__ inline void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// Counts kernel launches made by this library (reported by dcp_launch_count).
void note_launches(int64_t n);

inline int32_t launch_status(int64_t launches = 1) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return DCP_ERR_CUDA;
  note_launches(launches);
  return DCP_OK;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// cuTensorMapEncodeTiled from the driver, looked up once per process (nullptr if
// unavailable).  The function-local static is initialised under the C++ runtime's
// own lock, so concurrent first calls from several host threads are safe.
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

constexpr int kMaxDevices = 64;

// The current device, or -1 if it cannot be read or is kMaxDevices or above.
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// A kernel's dynamic shared-memory limit, raised on each device the first time
// a launch there needs more than the default (cudaFuncSetAttribute acts on the
// current device only).  One instance per kernel; safe to use from several host
// threads at once, e.g. one thread per GPU.
class SmemLimit {
 public:
  bool ensure(const void* kernel, size_t bytes) {
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lock(m_);
    if (set_[dev] >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
      return false;
    set_[dev] = bytes;
    return true;
  }

 private:
  std::mutex m_;
  size_t set_[kMaxDevices] = {};
};

}  // namespace dcp
