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

// ---------------------------------------------------------------- 512-dim rows, one warp per row
// Lane l owns the 16 dims [8l, 8l+8) and [256 + 8l, 256 + 8l + 8) of a 512-dim
// row in every dtype (so f32 and bf16 rows agree on which lane holds which
// dim); every warp access is one contiguous 1024-byte (f32) or 512-byte (bf16)
// segment.  Rows must be 16-byte aligned.
template <int kBf16>
__device__ inline const void* row_ptr(const void* base, int64_t row) {
  return static_cast<const unsigned char*>(base) + row * (int64_t)kDv * (kBf16 ? 2 : 4);
}
template <int kBf16>
__device__ inline void* row_ptr(void* base, int64_t row) {
  return static_cast<unsigned char*>(base) + row * (int64_t)kDv * (kBf16 ? 2 : 4);
}

template <int kInBf16>
__device__ inline void load16(const void* row, int lane, float (&v)[16]) {
  if (kInBf16) {
    const uint4* p = static_cast<const uint4*>(row);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint4 u = __ldg(p + lane + 32 * j);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f = __bfloat1622float2(h[k]);
        v[8 * j + 2 * k] = f.x;
        v[8 * j + 2 * k + 1] = f.y;
      }
    }
  } else {
    const float4* p = static_cast<const float4*>(row);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float4 a = __ldg(p + 2 * lane + 64 * j);
      float4 b = __ldg(p + 2 * lane + 64 * j + 1);
      v[8 * j + 0] = a.x; v[8 * j + 1] = a.y; v[8 * j + 2] = a.z; v[8 * j + 3] = a.w;
      v[8 * j + 4] = b.x; v[8 * j + 5] = b.y; v[8 * j + 6] = b.z; v[8 * j + 7] = b.w;
    }
  }
}

template <int kOutBf16>
__device__ inline void store16(void* row, int lane, const float (&v)[16]) {
  if (kOutBf16) {
    uint4* p = static_cast<uint4*>(row);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[8 * j + 2 * k], v[8 * j + 2 * k + 1]);
      p[lane + 32 * j] = u;
    }
  } else {
    float4* p = static_cast<float4*>(row);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      p[2 * lane + 64 * j] = make_float4(v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3]);
      p[2 * lane + 64 * j + 1] = make_float4(v[8 * j + 4], v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]);
    }
  }
}

// ---------------------------------------------------------------- all-to-all wire format
// One rank's send buffer holds, for each destination in turn, a chunk of
// a2a_chunk_bytes: an o block [n_held][rows][512] (bf16 or f32) and, at
// a2a_o_block_bytes, an lse block [n_held][rows] f32, padded to 256 bytes so
// that every chunk starts aligned.  rows = query tokens x heads per destination.
inline int64_t a2a_o_block_bytes(int64_t n_held, int64_t rows, int wire_bf16) {
  return n_held * rows * kDv * (wire_bf16 ? 2 : 4);
}
inline int64_t a2a_chunk_bytes(int64_t n_held, int64_t rows, int wire_bf16) {
  return (a2a_o_block_bytes(n_held, rows, wire_bf16) + n_held * rows * 4 + 255) & ~int64_t(255);
}

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
