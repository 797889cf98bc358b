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
// The same kernel merges the parts of an all-to-all receive buffer in place
// (dcp_lse_merge_packed): "Decode Context Parallelism" (zdszero), "通信策略",
// all-to-all form: the receiver holds its heads' partials of every shard and
// merges them locally.
#include "dcp_internal.cuh"

using namespace dcp;

namespace {

// Part r of merged row `row` in a dense [n_parts][rows] layout (dcp_lse_merge).
struct DenseParts {
  const void* o;
  const float* lse;
  int64_t rows;
  template <int kBf16>
  __device__ const void* o_row(int r, int64_t row) const {
    return row_ptr<kBf16>(o, (int64_t)r * rows + row);
  }
  __device__ float lse_at(int r, int64_t row) const { return __ldg(lse + (int64_t)r * rows + row); }
};

// Part r = w * n_held + s of merged row `row` in an all-to-all receive buffer
// (dcp_lse_merge_packed): chunk w came from rank w and holds its o block
// [n_held][rows][512] followed, at lse_off, by its lse block [n_held][rows].
struct PackedParts {
  const unsigned char* base;
  int64_t chunk, lse_off, rows;
  int32_t n_held;
  template <int kBf16>
  __device__ const void* o_row(int r, int64_t row) const {
    const int w = r / n_held, s = r - w * n_held;
    return row_ptr<kBf16>(base + w * chunk, (int64_t)s * rows + row);
  }
  __device__ float lse_at(int r, int64_t row) const {
    const int w = r / n_held, s = r - w * n_held;
    return __ldg(reinterpret_cast<const float*>(base + w * chunk + lse_off) + (int64_t)s * rows + row);
  }
};

template <class Parts, int kInBf16, int kOutBf16, int kBase2>
__global__ void __launch_bounds__(256) lse_merge_kernel(Parts parts, int32_t n_parts, int64_t rows,
                                                        void* __restrict__ o, float* __restrict__ lse) {
  const int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // pass 1: m = max_r lse_r
  float m = -INFINITY;
  for (int r = lane; r < n_parts; r += 32) m = fmaxf(m, parts.lse_at(r, row));
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  if (m == -INFINITY) {  // every part empty: the unit of the merge
    store16<kOutBf16>(row_ptr<kOutBf16>(o, row), lane, acc);
    if (lse && lane == 0) lse[row] = -INFINITY;
    return;
  }
  // pass 2: weights relative to m, weighted sum of the partial outputs
  float wsum = 0.f;
  for (int r = 0; r < n_parts; ++r) {
    const float l = parts.lse_at(r, row);
    if (l == -INFINITY) continue;  // zero weight; its o_r is not read
    const float w = kBase2 ? exp2f(l - m) : expf(l - m);
    wsum += w;
    float v[16];
    load16<kInBf16>(parts.template o_row<kInBf16>(r, row), lane, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = fmaf(w, v[i], acc[i]);
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] *= inv;
  store16<kOutBf16>(row_ptr<kOutBf16>(o, row), lane, acc);
  if (lse && lane == 0) lse[row] = m + (kBase2 ? log2f(wsum) : logf(wsum));
}

template <class Parts>
int32_t launch_merge(const Parts& parts, int32_t n, int64_t rows, int in_bf16, int out_bf16, int base2, void* o,
                     float* lse, void* stream) {
  const int64_t blocks = (rows + 7) / 8;  // 8 rows (warps) per block
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)blocks);
  cudaStream_t st = as_stream(stream);
  const int sel = in_bf16 * 4 + out_bf16 * 2 + base2;
  switch (sel) {
#define DCP_MERGE_CASE(I, O, B2) \
  case I * 4 + O * 2 + B2: lse_merge_kernel<Parts, I, O, B2><<<grid, 256, 0, st>>>(parts, n, rows, o, lse); break;
    DCP_MERGE_CASE(0, 0, 0) DCP_MERGE_CASE(0, 0, 1) DCP_MERGE_CASE(0, 1, 0) DCP_MERGE_CASE(0, 1, 1)
    DCP_MERGE_CASE(1, 0, 0) DCP_MERGE_CASE(1, 0, 1) DCP_MERGE_CASE(1, 1, 0) DCP_MERGE_CASE(1, 1, 1)
#undef DCP_MERGE_CASE
  }
  return launch_status();
}

bool dtype_ok(int32_t d) { return d == DCP_F32 || d == DCP_BF16; }

}  // namespace

extern "C" int32_t dcp_lse_merge(int32_t n_parts, int64_t rows, const void* o_part,
                                 int32_t o_part_dtype, const float* lse_part, int32_t lse_base,
                                 void* o, int32_t o_dtype, float* lse, void* stream) {
  if (n_parts < 1 || rows < 0) return DCP_ERR_INVALID;
  if (!dtype_ok(o_part_dtype) || !dtype_ok(o_dtype)) return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (rows == 0) return DCP_OK;
  if (!o_part || !lse_part || !o) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(o_part) | reinterpret_cast<uintptr_t>(o)) & 15) return DCP_ERR_INVALID;
  return launch_merge(DenseParts{o_part, lse_part, rows}, n_parts, rows, o_part_dtype == DCP_BF16,
                      o_dtype == DCP_BF16, lse_base == DCP_LSE_BASE_2, o, lse, stream);
}

extern "C" int32_t dcp_lse_merge_packed(int32_t world, int32_t n_held, int64_t rows, const void* recv,
                                        int32_t wire_dtype, int32_t lse_base, void* o, int32_t o_dtype, float* lse,
                                        void* stream) {
  if (world < 1 || n_held < 1 || rows < 0 || (int64_t)world * n_held > INT32_MAX) return DCP_ERR_INVALID;
  if (!dtype_ok(wire_dtype) || !dtype_ok(o_dtype)) return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (rows == 0) return DCP_OK;
  if (!recv || !o) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(recv) | reinterpret_cast<uintptr_t>(o)) & 15) return DCP_ERR_INVALID;
  const int wire_bf16 = wire_dtype == DCP_BF16;
  const PackedParts parts{static_cast<const unsigned char*>(recv), a2a_chunk_bytes(n_held, rows, wire_bf16),
                          a2a_o_block_bytes(n_held, rows, wire_bf16), rows, n_held};
  return launch_merge(parts, world * n_held, rows, wire_bf16, o_dtype == DCP_BF16, lse_base == DCP_LSE_BASE_2, o,
                      lse, stream);
}
