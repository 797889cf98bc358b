// dcp_layout.cu — slot map, owner-filtered append and prefill-to-decode
// relayout (integer / copy kernels).
//
// dcp_slot_map: one thread per new token computes (owner, local row, slot).
// dcp_kv_append: one warp per new token computes the same placement and copies
// its 1152-byte latent row with 16-byte vector loads/stores into the owner's
// pool.  Both are tiny next to the decode partial (B tokens per decode step;
// 8192 per chunk), so they are written for latency: one launch, no shared
// memory.
// dcp_kv_relayout: one warp per listed token of a paged prefill pool: owner
// filter, source and destination rows, a 1152-byte copy (HBM-bound for long
// requests: 2 x 1152 bytes per moved token).
#include "dcp_internal.cuh"

#include <atomic>

using namespace dcp;

namespace dcp {
static std::atomic<int64_t> g_launches{0};
void note_launches(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace dcp

extern "C" int64_t dcp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int32_t dcp_version(void) { return 10000; }

extern "C" const char* dcp_error_string(int32_t code) {
  switch (code) {
    case DCP_OK: return "ok";
    case DCP_ERR_INVALID: return "invalid argument";
    case DCP_ERR_UNSUPPORTED: return "unsupported configuration";
    case DCP_ERR_CUDA: return "CUDA call failed";
    case DCP_ERR_WORKSPACE: return "workspace missing or too small";
    case DCP_ERR_TOO_LARGE: return "sizes need more scratch than the built-in area";
    default: return "unknown error";
  }
}

extern "C" int64_t dcp_count(const dcp_layout_t* layout, int32_t shard, int64_t x) {
  if (!layout_ok(layout) || shard < 0 || shard >= layout->n_shards || x < 0) return -1;
  return count_of(shard, x, to_layout(layout));
}

namespace {

__global__ void slot_map_kernel(Layout L, const int64_t* __restrict__ pos,
                                const int32_t* __restrict__ req, int64_t T,
                                const int32_t* __restrict__ bt, int32_t B, int64_t bt_stride,
                                int64_t max_pages, int64_t pool_pages, int32_t* __restrict__ owner,
                                int64_t* __restrict__ row, int64_t* __restrict__ slot,
                                int32_t* status) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int64_t p = pos[t];
  const int32_t b = req[t];
  int64_t own = -1, r = -1, s = -1;
  if (p < 0) {
    flag(status, DCP_STATUS_BAD_POSITION);
  } else {
    own = owner_of(p, L);
    r = local_row_of(p, L);
    const int64_t page_idx = r / L.P;
    if (b < 0 || b >= B) {
      flag(status, DCP_STATUS_BAD_REQUEST);
    } else if (page_idx >= max_pages) {
      flag(status, DCP_STATUS_BAD_PAGE_INDEX);
    } else {
      const int64_t page = bt[(int64_t)b * bt_stride + page_idx];
      if (page < 0 || page >= pool_pages) {
        flag(status, DCP_STATUS_BAD_PAGE_ID);
      } else {
        s = page * L.P + r % L.P;
      }
    }
  }
  owner[t] = (int32_t)own;
  row[t] = r;
  slot[t] = s;
}

// Owner-filtered append: one warp per new token.  Every lane computes the
// token's owner, local row and slot (the slot map's formulas), so the copy needs
// no separate slot-map launch; tokens of shards this call does not hold stop
// before reading their block-table entry.  The 1152-byte row moves as 72
// 16-byte vectors.  Positions below 2^31 take 32-bit index math.
__global__ void kv_append_kernel(Layout L, int32_t shard_begin, int32_t shard_end, const uint4* __restrict__ kv_new,
                                 const int64_t* __restrict__ pos, const int32_t* __restrict__ req, int64_t T,
                                 const int32_t* __restrict__ bt, int32_t B, int64_t bt_stride, int64_t max_pages,
                                 uint4* __restrict__ arena, int64_t pool_pages, int32_t* status) {
  constexpr int kVec = kDk * 2 / 16;  // 72
  const int64_t t = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t p = __ldg(pos + t);
  const int32_t b = __ldg(req + t);
  if (p < 0 || b < 0 || b >= B) {
    if (lane == 0) flag(status, p < 0 ? DCP_STATUS_BAD_POSITION : DCP_STATUS_BAD_REQUEST);
    return;
  }
  int64_t own, row;
  if (p < INT32_MAX) {
    const int32_t p32 = (int32_t)p, blk = p32 / L.I;
    own = blk % L.N;
    row = (int64_t)(blk / L.N) * L.I + p32 % L.I;
  } else {
    own = owner_of(p, L);
    row = local_row_of(p, L);
  }
  if (own < shard_begin || own >= shard_end) return;  // another device's shard
  // the row's loads go out before the block-table lookup, so the two latencies
  // overlap (the row is read whether or not its page turns out valid)
  const uint4* src = kv_new + t * kVec;
  uint4 v0 = __ldg(src + lane), v1 = __ldg(src + 32 + lane), v2 = make_uint4(0, 0, 0, 0);
  if (lane < kVec - 64) v2 = __ldg(src + 64 + lane);
  const int64_t pidx = row / L.P;
  if (pidx >= max_pages) {
    if (lane == 0) flag(status, DCP_STATUS_BAD_PAGE_INDEX);
    return;
  }
  const int64_t page = __ldg(bt + (int64_t)b * bt_stride + pidx);
  if (page < 0 || page >= pool_pages) {
    if (lane == 0) flag(status, DCP_STATUS_BAD_PAGE_ID);
    return;
  }
  const int64_t slot = page * L.P + row % L.P;
  uint4* dst = arena + ((own - shard_begin) * pool_pages * L.P + slot) * kVec;
  dst[lane] = v0;
  dst[32 + lane] = v1;
  if (lane < kVec - 64) dst[64 + lane] = v2;
}

// Prefill-to-decode relayout: one warp per listed token.  The owner filter
// runs before any read, so tokens of other shards cost only their indices.
// Positions below 2^31 (every realistic context) take 32-bit index math.
__global__ void kv_relayout_kernel(Layout L, int32_t shard_begin, int32_t shard_end, const uint4* __restrict__ src,
                                   int64_t src_rows, int32_t Ps, const int32_t* __restrict__ src_bt,
                                   int64_t src_bt_stride, int64_t src_max_pages, const int64_t* __restrict__ pos,
                                   const int32_t* __restrict__ req, int64_t T, int32_t B,
                                   const int32_t* __restrict__ bt, int64_t bt_stride, int64_t max_pages,
                                   uint4* __restrict__ arena, int64_t pool_rows, int32_t* status) {
  constexpr int kVec = kDk * 2 / 16;  // 72 16-byte pieces per row
  const int64_t t = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t p = __ldg(pos + t);
  const int32_t b = __ldg(req + t);
  if (p < 0 || b < 0 || b >= B) {
    if (lane == 0) flag(status, p < 0 ? DCP_STATUS_BAD_POSITION : DCP_STATUS_BAD_REQUEST);
    return;
  }
  int64_t own, row, src_pidx, src_off;
  if (p < INT32_MAX) {
    const int32_t p32 = (int32_t)p, blk = p32 / L.I;
    own = blk % L.N;
    row = (int64_t)(blk / L.N) * L.I + p32 % L.I;
    src_pidx = p32 / Ps;
    src_off = p32 % Ps;
  } else {
    own = owner_of(p, L);
    row = local_row_of(p, L);
    src_pidx = p / Ps;
    src_off = p % Ps;
  }
  if (own < shard_begin || own >= shard_end) return;  // another device's shard
  const int64_t pidx = row / L.P;
  if (src_pidx >= src_max_pages || pidx >= max_pages) {
    if (lane == 0) flag(status, DCP_STATUS_BAD_PAGE_INDEX);
    return;
  }
  const int64_t sp = __ldg(src_bt + (int64_t)b * src_bt_stride + src_pidx);
  const int64_t dp = __ldg(bt + (int64_t)b * bt_stride + pidx);
  const int64_t srow = sp * Ps + src_off, drow = dp * L.P + row % L.P;
  if (sp < 0 || srow >= src_rows || dp < 0 || drow >= pool_rows) {
    if (lane == 0) flag(status, DCP_STATUS_BAD_PAGE_ID);
    return;
  }
  const uint4* s = src + srow * kVec;
  uint4* d = arena + ((int64_t)(own - shard_begin) * pool_rows + drow) * kVec;
  uint4 v0 = __ldg(s + lane), v1 = __ldg(s + 32 + lane), v2;
  if (lane < kVec - 64) v2 = __ldg(s + 64 + lane);
  d[lane] = v0;
  d[32 + lane] = v1;
  if (lane < kVec - 64) d[64 + lane] = v2;
}

}  // namespace

extern "C" int32_t dcp_kv_relayout(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                                   const void* src_pool, int64_t src_pool_rows, int32_t src_page_size,
                                   const int32_t* src_block_table, int64_t src_bt_stride, int64_t src_max_pages,
                                   const int64_t* pos, const int32_t* req, int64_t T, int32_t B,
                                   const int32_t* block_table, int64_t bt_stride, int64_t max_pages, void* arena,
                                   int64_t pool_pages, int32_t* status, void* stream) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end ||
      T < 0 || B < 1 || src_page_size < 1 || src_pool_rows < 1 || pool_pages < 1 || src_max_pages < 1 ||
      src_bt_stride < src_max_pages || max_pages < 1 || bt_stride < max_pages)
    return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!src_pool || !src_block_table || !pos || !req || !block_table || !arena || !status) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(src_pool) | reinterpret_cast<uintptr_t>(arena)) & 15)
    return DCP_ERR_INVALID;  // rows are moved as 16-byte vectors
  const int threads = 256;  // 8 tokens per block
  const int64_t blocks = (T * 32 + threads - 1) / threads;
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  kv_relayout_kernel<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(
      to_layout(layout), shard_begin, shard_end, static_cast<const uint4*>(src_pool), src_pool_rows, src_page_size,
      src_block_table, src_bt_stride, src_max_pages, pos, req, T, B, block_table, bt_stride, max_pages,
      static_cast<uint4*>(arena), pool_pages * layout->page_size, status);
  return launch_status();
}

extern "C" int32_t dcp_slot_map(const dcp_layout_t* layout, const int64_t* pos, const int32_t* req,
                                int64_t T, const int32_t* block_table, int32_t B, int64_t bt_stride,
                                int64_t max_pages, int64_t pool_pages, int32_t* owner, int64_t* row,
                                int64_t* slot, int32_t* status, void* stream) {
  if (!layout_ok(layout) || T < 0 || B < 1 || max_pages < 1 || bt_stride < max_pages ||
      pool_pages < 1)
    return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!pos || !req || !block_table || !owner || !row || !slot) return DCP_ERR_INVALID;
  const int threads = 256;
  const int64_t blocks = (T + threads - 1) / threads;
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  slot_map_kernel<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(
      to_layout(layout), pos, req, T, block_table, B, bt_stride, max_pages, pool_pages, owner, row,
      slot, status);
  return launch_status();
}

extern "C" int32_t dcp_kv_append(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                                 const void* kv_new, const int64_t* pos, const int32_t* req, int64_t T,
                                 const int32_t* block_table, int32_t B, int64_t bt_stride, int64_t max_pages,
                                 void* arena, int64_t pool_pages, int32_t* status, void* stream) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end || T < 0 ||
      B < 1 || max_pages < 1 || bt_stride < max_pages || pool_pages < 1)
    return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!kv_new || !pos || !req || !block_table || !arena) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(kv_new) | reinterpret_cast<uintptr_t>(arena)) & 15)
    return DCP_ERR_INVALID;  // rows are moved as 16-byte vectors
  const int threads = 256;  // 8 tokens per block
  const int64_t blocks = (T * 32 + threads - 1) / threads;
  if (blocks > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  kv_append_kernel<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(
      to_layout(layout), shard_begin, shard_end, static_cast<const uint4*>(kv_new), pos, req, T, block_table, B,
      bt_stride, max_pages, static_cast<uint4*>(arena), pool_pages, status);
  return launch_status();
}
