// dcp_decode.cu — per-shard partial attention (o_r, lse_r) for absorbed MLA.
//
// Sources: "MLA 的 Decode Context Parallelism", section 2 (absorbed form: one
// 576-d KV head shared by all query heads; values are the first 512 dims) and
// section 3 (each rank returns its locally normalised output and its LSE);
// "Decode Context Parallelism" (zdszero), "Core abstraction" idea 2;
// SGLang "Decode context parallelism", "DCP x speculative decoding" (causal
// mask in global positions, from the shard rank and the global lengths).
//
// First version: a plain SIMT kernel, one CTA per (16 query rows, shard,
// request), streaming the shard's rows through shared memory in tiles of 32
// with an online (running max / running sum) softmax.  Visible local rows of
// query row (t, h): [0, count_r(S_b - q_len + t + 1)).
#include "dcp_internal.cuh"

using namespace dcp;

namespace {

constexpr int kRowsPerCta = 16;
constexpr int kTile = 32;
constexpr int kKvPitch = kDk + 8;  // bf16 elements; 1168-byte rows stay 16-byte aligned
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct PartialArgs {
  Layout L;
  int32_t shard_begin;
  const __nv_bfloat16* q;
  int32_t B, q_len, H;
  const __nv_bfloat16* arena;
  int64_t pool_rows;
  int64_t pool_pages;
  const int32_t* bt;
  int64_t bt_stride, max_pages;
  const int64_t* seq_lens;
  float scale_log2;  // scale * log2(e): scores are kept in base 2
  int32_t base2;
  void* o_part;
  int32_t o_bf16;
  float* lse_part;
  int32_t* status;
};

__global__ void __launch_bounds__(256) partial_simt_kernel(PartialArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* q_s = reinterpret_cast<float*>(smem);                                       // [16][576]
  __nv_bfloat16* kv_s = reinterpret_cast<__nv_bfloat16*>(q_s + kRowsPerCta * kDk);  // [32][580]
  __shared__ int64_t nvis_s[kRowsPerCta];

  const int tid = threadIdx.x;
  const int i = tid >> 4;   // row within the CTA
  const int j = tid & 15;   // lane within the row group
  const int R = a.q_len * a.H;
  const int row0 = blockIdx.x * kRowsPerCta;
  const int rs = blockIdx.y;              // held-shard index
  const int64_t r = a.shard_begin + rs;   // global shard id
  const int b = blockIdx.z;
  const int64_t S = a.seq_lens[b];
  const bool bad_len = S < a.q_len;
  if (bad_len && tid == 0) flag(a.status, DCP_STATUS_BAD_LENGTH);

  // query rows -> fp32 in shared memory; visible-row count per query row
  for (int e = tid; e < kRowsPerCta * kDk; e += blockDim.x) {
    const int ri = e / kDk, d = e % kDk;
    const int row = row0 + ri;
    float v = 0.f;
    if (row < R) v = __bfloat162float(a.q[((int64_t)b * R + row) * kDk + d]);
    q_s[e] = v;
  }
  if (tid < kRowsPerCta) {
    const int row = row0 + tid;
    int64_t nv = 0;
    if (row < R && !bad_len) {
      const int t = row / a.H;
      nv = count_of(r, S - a.q_len + t + 1, a.L);
    }
    nvis_s[tid] = nv;
  }
  __syncthreads();
  int64_t n_max = 0;
  for (int k = 0; k < kRowsPerCta; ++k) n_max = max(n_max, nvis_s[k]);
  const int64_t my_nvis = nvis_s[i];

  float m = -INFINITY;  // running max (base-2 units)
  float l = 0.f;        // running sum of exp2(s - m)
  float acc[32];        // dims 2*(j + 16k) and +1, k = 0..15
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.f;

  const __nv_bfloat16* pool = a.arena + (int64_t)rs * a.pool_rows * kDk;
  const int32_t* bt_b = a.bt + (int64_t)b * a.bt_stride;

  for (int64_t rho0 = 0; rho0 < n_max; rho0 += kTile) {
    __syncthreads();
    // gather 32 local rows through the block table (16-byte vectors)
    for (int e = tid; e < kTile * (kDk / 8); e += blockDim.x) {
      const int tr = e / (kDk / 8), c = e % (kDk / 8);
      const int64_t rho = rho0 + tr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (rho < n_max) {
        const int64_t pidx = rho / a.L.P;
        const int64_t page = pidx < a.max_pages ? (int64_t)bt_b[pidx] : -1;
        if (page >= 0 && page < a.pool_pages) {
          v = __ldg(reinterpret_cast<const uint4*>(pool + (page * a.L.P + rho % a.L.P) * kDk) + c);
        } else if (c == 0) {
          flag(a.status, DCP_STATUS_BAD_PAGE_ID);
        }
      }
      *reinterpret_cast<uint4*>(kv_s + tr * kKvPitch + c * 8) = v;
    }
    __syncthreads();
    // scores of tokens j and j+16 for row i
    float s[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int tok = j + 16 * u;
      const __nv_bfloat162* kr = reinterpret_cast<const __nv_bfloat162*>(kv_s + tok * kKvPitch);
      const float2* qr = reinterpret_cast<const float2*>(q_s + i * kDk);
      float dot = 0.f;
#pragma unroll 8
      for (int d2 = 0; d2 < kDk / 2; ++d2) {
        const float2 kf = __bfloat1622float2(kr[d2]);
        const float2 qf = qr[d2];
        dot = fmaf(qf.x, kf.x, dot);
        dot = fmaf(qf.y, kf.y, dot);
      }
      s[u] = (rho0 + tok < my_nvis) ? dot * a.scale_log2 : -INFINITY;
    }
    float tmax = fmaxf(s[0], s[1]);
#pragma unroll
    for (int sh = 8; sh > 0; sh >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, sh));
    const float m_new = fmaxf(m, tmax);
    float p[2] = {0.f, 0.f};
    float alpha = 1.f;
    if (m_new != -INFINITY) {
      alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
      p[0] = exp2f(s[0] - m_new);
      p[1] = exp2f(s[1] - m_new);
    }
    float psum = p[0] + p[1];
#pragma unroll
    for (int sh = 8; sh > 0; sh >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, sh);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] *= alpha;
    const int grp = (tid & 31) & 16;  // lane offset of this row's 16-lane group
    for (int tok = 0; tok < kTile; ++tok) {
      const float pt = __shfl_sync(0xffffffffu, p[tok >> 4], grp + (tok & 15));
      const __nv_bfloat162* vr = reinterpret_cast<const __nv_bfloat162*>(kv_s + tok * kKvPitch);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 vf = __bfloat1622float2(vr[j + 16 * k]);
        acc[2 * k] = fmaf(pt, vf.x, acc[2 * k]);
        acc[2 * k + 1] = fmaf(pt, vf.y, acc[2 * k + 1]);
      }
    }
  }

  const int row = row0 + i;
  if (row >= R) return;
  const int64_t out_row = ((int64_t)rs * a.B + b) * R + row;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (a.o_bf16) {
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(a.o_part) + out_row * kDv);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[j + 16 * k] = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
  } else {
    float2* o = reinterpret_cast<float2*>(static_cast<float*>(a.o_part) + out_row * kDv);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[j + 16 * k] = make_float2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
  }
  if (j == 0) {
    float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
    a.lse_part[out_row] = a.base2 ? lse2 : lse2 * kLn2;
  }
}

constexpr size_t kSmemBytes = kRowsPerCta * kDk * sizeof(float) + kTile * kKvPitch * sizeof(__nv_bfloat16);

}  // namespace

extern "C" size_t dcp_mla_decode_workspace_size(const dcp_layout_t* layout, int32_t shard_begin,
                                                int32_t shard_end, int32_t B, int32_t q_len, int32_t H) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end ||
      B < 1 || q_len < 1 || H < 1)
    return 0;
  return 0;
}

extern "C" int32_t dcp_mla_decode_partial(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                                          const void* q, int32_t B, int32_t q_len, int32_t H,
                                          const void* arena, int64_t pool_pages,
                                          const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                                          const int64_t* seq_lens, float scale, int32_t lse_base,
                                          void* o_part, int32_t o_part_dtype, float* lse_part,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* status, void* stream) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end)
    return DCP_ERR_INVALID;
  if (B < 1 || q_len < 1 || H < 1 || (int64_t)q_len * H > 1024) return DCP_ERR_INVALID;
  if (pool_pages < 1 || max_pages < 1 || bt_stride < max_pages) return DCP_ERR_INVALID;
  if (!q || !arena || !block_table || !seq_lens || !o_part || !lse_part) return DCP_ERR_INVALID;
  if (o_part_dtype != DCP_F32 && o_part_dtype != DCP_BF16) return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (!(scale > 0.f) || !(scale < INFINITY)) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(arena) |
       reinterpret_cast<uintptr_t>(o_part)) & 15)
    return DCP_ERR_INVALID;
  const size_t need = dcp_mla_decode_workspace_size(layout, shard_begin, shard_end, B, q_len, H);
  if (workspace_bytes < need || (need > 0 && !workspace)) return DCP_ERR_WORKSPACE;

  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(partial_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return DCP_ERR_CUDA;
    attr_set = true;
  }
  PartialArgs a;
  a.L = to_layout(layout);
  a.shard_begin = shard_begin;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.B = B; a.q_len = q_len; a.H = H;
  a.arena = static_cast<const __nv_bfloat16*>(arena);
  a.pool_pages = pool_pages;
  a.pool_rows = pool_pages * layout->page_size;
  a.bt = block_table; a.bt_stride = bt_stride; a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.scale_log2 = scale * kLog2e;
  a.base2 = lse_base == DCP_LSE_BASE_2;
  a.o_part = o_part; a.o_bf16 = o_part_dtype == DCP_BF16;
  a.lse_part = lse_part;
  a.status = status;
  const int R = q_len * H;
  dim3 grid((R + kRowsPerCta - 1) / kRowsPerCta, shard_end - shard_begin, B);
  if (B > 65535) return DCP_ERR_UNSUPPORTED;
  partial_simt_kernel<<<grid, 256, kSmemBytes, as_stream(stream)>>>(a);
  return launch_status();
}
