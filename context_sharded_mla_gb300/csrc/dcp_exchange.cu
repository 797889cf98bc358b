// dcp_exchange.cu — the cross-rank side of the partials: packing them by head
// slice for the all-to-all, and the local step of the AllGather + ReduceScatter
// merge.  Both are HBM-bound row copies, one warp per 512-dim row.
//
// Sources: "Decode Context Parallelism" (zdszero), section "通信策略":
//  - "合并：All-to-All": each rank cuts O_r by head into one piece per rank and
//    sends it, with the matching LSE in the same buffer, to the rank that owns
//    those heads (one collective per layer);
//  - "合并：AllGather + ReduceScatter": all ranks' LSE are gathered, each rank
//    forms the global L and corrects its partial to exp(L_r - L) O_r, and a
//    reduce-scatter sums the corrected partials and scatters them by head.
// "MLA 的 Decode Context Parallelism", section 4, stages 6-7 (all-to-all of
// (o^(r), lse_r) to the head owner, then the two-pass merge there).
//
// Rank w holds shards [w * n_held, (w + 1) * n_held) and owns heads
// [w * Hd, (w + 1) * Hd), Hd = H / world.  The partials of a rank are
// o_part [n_held][T][H][512] and lse_part [n_held][T][H] (T query tokens).
#include "dcp_internal.cuh"

using namespace dcp;

namespace {

// One warp per partial row (s, t, h): its o row goes, in the wire dtype, to row
// (s, t, h % Hd) of destination h / Hd's o block, its lse to the same row of
// that chunk's lse block.
template <int kInBf16, int kWireBf16>
__global__ void __launch_bounds__(256) pack_kernel(int32_t n_held, int32_t T, int32_t H, int32_t Hd,
                                                   const void* __restrict__ o_part, const float* __restrict__ lse_part,
                                                   unsigned char* __restrict__ send, int64_t chunk, int64_t lse_off) {
  const int64_t i = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;  // (s * T + t) * H + h
  const int lane = threadIdx.x & 31;
  if (i >= (int64_t)n_held * T * H) return;
  const int64_t st = i / H;  // s * T + t
  const int h = (int)(i - st * H);
  const int d = h / Hd;
  const int64_t drow = st * Hd + (h - d * Hd);  // row inside destination d's blocks
  unsigned char* dst = send + d * chunk;
  float v[16];
  load16<kInBf16>(row_ptr<kInBf16>(o_part, i), lane, v);
  store16<kWireBf16>(row_ptr<kWireBf16>(dst, drow), lane, v);
  if (lane == 0) reinterpret_cast<float*>(dst + lse_off)[drow] = __ldg(lse_part + i);
}

// AllGather + ReduceScatter, local step: one warp per row (t, h).  lse_all holds
// the lse of every shard in shard order [n_shards][T * H]; the row's global
// L = m + log sum_r base^(lse_r - m); this rank's corrected sum
// sum_{s held} base^(lse_{shard_begin + s} - L) o_part[s] is written, f32, to row
// (t, h % Hd) of block h / Hd of o_sum [world][T][Hd][512], and L to the same
// place of lse_out [world][T][Hd].  A row whose shards are all empty gets 0 and
// -inf; an empty held shard has zero weight and its o row is not read.
template <int kInBf16, int kBase2>
__global__ void __launch_bounds__(256) rescale_kernel(int32_t n_shards, int32_t shard_begin, int32_t n_held, int32_t T,
                                                      int32_t H, int32_t Hd, const float* __restrict__ lse_all,
                                                      const void* __restrict__ o_part, float* __restrict__ o_sum,
                                                      float* __restrict__ lse_out) {
  const int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;  // t * H + h
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)T * H;
  if (row >= rows) return;
  const int64_t t = row / H;
  const int h = (int)(row - t * H);
  const int d = h / Hd;
  const int64_t drow = ((int64_t)d * T + t) * Hd + (h - d * Hd);
  float m = -INFINITY;
  for (int r = lane; r < n_shards; r += 32) m = fmaxf(m, __ldg(lse_all + (int64_t)r * rows + row));
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float L = -INFINITY;
  if (m != -INFINITY) {
    float z = 0.f;  // lanes share the shards; every lane ends with the full sum
    for (int r = lane; r < n_shards; r += 32) {
      const float l = __ldg(lse_all + (int64_t)r * rows + row);
      if (l != -INFINITY) z += kBase2 ? exp2f(l - m) : expf(l - m);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) z += __shfl_xor_sync(0xffffffffu, z, s);
    L = m + (kBase2 ? log2f(z) : logf(z));
    for (int s = 0; s < n_held; ++s) {
      const float l = __ldg(lse_all + (int64_t)(shard_begin + s) * rows + row);
      if (l == -INFINITY) continue;
      const float w = kBase2 ? exp2f(l - L) : expf(l - L);
      float v[16];
      load16<kInBf16>(row_ptr<kInBf16>(o_part, (int64_t)s * rows + row), lane, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = fmaf(w, v[i], acc[i]);
    }
  }
  store16<0>(row_ptr<0>(o_sum, drow), lane, acc);
  if (lse_out && lane == 0) lse_out[drow] = L;
}

bool dtype_ok(int32_t d) { return d == DCP_F32 || d == DCP_BF16; }

bool split_ok(int32_t n_held, int32_t T, int32_t H, int32_t world) {
  return n_held >= 1 && T >= 0 && H >= 1 && world >= 1 && H % world == 0 &&
         (int64_t)n_held * T * H < ((int64_t)1 << 40);
}

}  // namespace

extern "C" size_t dcp_a2a_chunk_bytes(int32_t n_held, int32_t T, int32_t H, int32_t world, int32_t wire_dtype) {
  if (!split_ok(n_held, T, H, world) || !dtype_ok(wire_dtype)) return 0;
  return (size_t)a2a_chunk_bytes(n_held, (int64_t)T * (H / world), wire_dtype == DCP_BF16);
}

extern "C" int32_t dcp_pack_partials(int32_t n_held, int32_t T, int32_t H, int32_t world, const void* o_part,
                                     int32_t o_part_dtype, const float* lse_part, void* send, int32_t wire_dtype,
                                     void* stream) {
  if (!split_ok(n_held, T, H, world) || !dtype_ok(o_part_dtype) || !dtype_ok(wire_dtype)) return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!o_part || !lse_part || !send) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(o_part) | reinterpret_cast<uintptr_t>(send)) & 15) return DCP_ERR_INVALID;
  const int Hd = H / world;
  const int wb = wire_dtype == DCP_BF16;
  const int64_t rows_d = (int64_t)T * Hd;
  const int64_t chunk = a2a_chunk_bytes(n_held, rows_d, wb), lse_off = a2a_o_block_bytes(n_held, rows_d, wb);
  const int64_t blocks = ((int64_t)n_held * T * H + 7) / 8;
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  unsigned char* out = static_cast<unsigned char*>(send);
  const bool ib = o_part_dtype == DCP_BF16;
  if (ib && wb)
    pack_kernel<1, 1><<<(unsigned)blocks, 256, 0, st>>>(n_held, T, H, Hd, o_part, lse_part, out, chunk, lse_off);
  else if (ib)
    pack_kernel<1, 0><<<(unsigned)blocks, 256, 0, st>>>(n_held, T, H, Hd, o_part, lse_part, out, chunk, lse_off);
  else if (wb)
    pack_kernel<0, 1><<<(unsigned)blocks, 256, 0, st>>>(n_held, T, H, Hd, o_part, lse_part, out, chunk, lse_off);
  else
    pack_kernel<0, 0><<<(unsigned)blocks, 256, 0, st>>>(n_held, T, H, Hd, o_part, lse_part, out, chunk, lse_off);
  return launch_status();
}

extern "C" int32_t dcp_lse_rescale(int32_t n_shards, int32_t shard_begin, int32_t n_held, int32_t T, int32_t H,
                                   int32_t world, const float* lse_all, const void* o_part, int32_t o_part_dtype,
                                   int32_t lse_base, float* o_sum, float* lse, void* stream) {
  if (!split_ok(n_held, T, H, world) || !dtype_ok(o_part_dtype)) return DCP_ERR_INVALID;
  if (n_shards < 1 || shard_begin < 0 || shard_begin + n_held > n_shards) return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!lse_all || !o_part || !o_sum) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(o_part) | reinterpret_cast<uintptr_t>(o_sum)) & 15) return DCP_ERR_INVALID;
  const int64_t blocks = ((int64_t)T * H + 7) / 8;
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  const int Hd = H / world;
  const bool ib = o_part_dtype == DCP_BF16, b2 = lse_base == DCP_LSE_BASE_2;
  if (ib && b2)
    rescale_kernel<1, 1><<<(unsigned)blocks, 256, 0, st>>>(n_shards, shard_begin, n_held, T, H, Hd, lse_all, o_part,
                                                           o_sum, lse);
  else if (ib)
    rescale_kernel<1, 0><<<(unsigned)blocks, 256, 0, st>>>(n_shards, shard_begin, n_held, T, H, Hd, lse_all, o_part,
                                                           o_sum, lse);
  else if (b2)
    rescale_kernel<0, 1><<<(unsigned)blocks, 256, 0, st>>>(n_shards, shard_begin, n_held, T, H, Hd, lse_all, o_part,
                                                           o_sum, lse);
  else
    rescale_kernel<0, 0><<<(unsigned)blocks, 256, 0, st>>>(n_shards, shard_begin, n_held, T, H, Hd, lse_all, o_part,
                                                           o_sum, lse);
  return launch_status();
}
