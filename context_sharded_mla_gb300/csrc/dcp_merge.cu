// dcp_merge.cu — exact LSE merge of n partials (HBM-bound, vectorised).
//
// Sources: "Decode Context Parallelism" (zdszero), "Theory": the merge
// identity O = sum_r exp(L_r) O_r / sum_r exp(L_r) and its stable form with
// m = max_r L_r; the exp/log pair must match the base of the partials.
// "MLA 的 Decode Context Parallelism", section 3: w_r = exp2(lse_r - m),
// out = sum_r w_r o_r / sum_r w_r.
//
// One warp per output row.  Every lane owns 16 of the 512 value dims, read as
// 16-byte vectors so that each warp access is one contiguous 1024-byte (f32) or
// 512-byte (bf16) segment per part.  Algorithmic bytes per row:
// n_parts * (512 * sizeof(o_part) + 4) read, 512 * sizeof(o) + 4 written.
#include "dcp_internal.cuh"

using namespace dcp;

namespace {

// Lane l owns the 16 dims [8l, 8l+8) and [256 + 8l, 256 + 8l + 8) in every
// dtype, so the f32 and bf16 paths agree on which lane holds which dim.
template <int kInBf16>
__device__ inline void load16(const void* base, int64_t row, int lane, float (&v)[16]) {
  if (kInBf16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + row * kDv);
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
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * kDv);
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
__device__ inline void store16(void* base, int64_t row, int lane, const float (&v)[16]) {
  if (kOutBf16) {
    uint4* p = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row * kDv);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[8 * j + 2 * k], v[8 * j + 2 * k + 1]);
      p[lane + 32 * j] = u;
    }
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + row * kDv);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      p[2 * lane + 64 * j] = make_float4(v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3]);
      p[2 * lane + 64 * j + 1] = make_float4(v[8 * j + 4], v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]);
    }
  }
}

template <int kInBf16, int kOutBf16, int kBase2>
__global__ void __launch_bounds__(256) lse_merge_kernel(int32_t n_parts, int64_t rows,
                                                        const void* __restrict__ o_part,
                                                        const float* __restrict__ lse_part,
                                                        void* __restrict__ o, float* __restrict__ lse) {
  const int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // pass 1: m = max_r lse_r
  float m = -INFINITY;
  for (int r = lane; r < n_parts; r += 32) m = fmaxf(m, __ldg(lse_part + (int64_t)r * rows + row));
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  if (m == -INFINITY) {  // every part empty: the unit of the merge
    store16<kOutBf16>(o, row, lane, acc);
    if (lse && lane == 0) lse[row] = -INFINITY;
    return;
  }
  // pass 2: weights relative to m, weighted sum of the partial outputs
  float wsum = 0.f;
  for (int r = 0; r < n_parts; ++r) {
    const float l = __ldg(lse_part + (int64_t)r * rows + row);
    if (l == -INFINITY) continue;  // zero weight; its o_r is not read
    const float w = kBase2 ? exp2f(l - m) : expf(l - m);
    wsum += w;
    float v[16];
    load16<kInBf16>(o_part, (int64_t)r * rows + row, lane, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = fmaf(w, v[i], acc[i]);
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] *= inv;
  store16<kOutBf16>(o, row, lane, acc);
  if (lse && lane == 0) lse[row] = m + (kBase2 ? log2f(wsum) : logf(wsum));
}

template <int kInBf16, int kOutBf16>
void launch_merge(int base2, dim3 grid, cudaStream_t st, int32_t n, int64_t rows, const void* op,
                  const float* lp, void* o, float* lse) {
  if (base2)
    lse_merge_kernel<kInBf16, kOutBf16, 1><<<grid, 256, 0, st>>>(n, rows, op, lp, o, lse);
  else
    lse_merge_kernel<kInBf16, kOutBf16, 0><<<grid, 256, 0, st>>>(n, rows, op, lp, o, lse);
}

}  // namespace

extern "C" int32_t dcp_lse_merge(int32_t n_parts, int64_t rows, const void* o_part,
                                 int32_t o_part_dtype, const float* lse_part, int32_t lse_base,
                                 void* o, int32_t o_dtype, float* lse, void* stream) {
  if (n_parts < 1 || rows < 0) return DCP_ERR_INVALID;
  if ((o_part_dtype != DCP_F32 && o_part_dtype != DCP_BF16) || (o_dtype != DCP_F32 && o_dtype != DCP_BF16))
    return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (rows == 0) return DCP_OK;
  if (!o_part || !lse_part || !o) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(o_part) | reinterpret_cast<uintptr_t>(o)) & 15) return DCP_ERR_INVALID;
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)blocks);
  cudaStream_t st = as_stream(stream);
  const int b2 = lse_base == DCP_LSE_BASE_2;
  if (o_part_dtype == DCP_BF16) {
    if (o_dtype == DCP_BF16) launch_merge<1, 1>(b2, grid, st, n_parts, rows, o_part, lse_part, o, lse);
    else launch_merge<1, 0>(b2, grid, st, n_parts, rows, o_part, lse_part, o, lse);
  } else {
    if (o_dtype == DCP_BF16) launch_merge<0, 1>(b2, grid, st, n_parts, rows, o_part, lse_part, o, lse);
    else launch_merge<0, 0>(b2, grid, st, n_parts, rows, o_part, lse_part, o, lse);
  }
  return launch_status();
}
