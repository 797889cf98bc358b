// dcp_decode.cu — per-shard partial attention (o_r, lse_r) for absorbed MLA on sm_103a.
//
// Sources: "MLA 的 Decode Context Parallelism", section 2 (absorbed form: one
// 576-d KV head shared by all query heads; values are the first 512 dims) and
// section 3 (each rank returns its locally normalised output and its LSE);
// "Decode Context Parallelism" (zdszero), "Core abstraction" idea 2 and
// "Theory" (the (Z, N) merge operator: a shard may itself be split into pieces
// that are merged the same way); SGLang "Decode context parallelism",
// "DCP x speculative decoding" (causal mask in global positions, from the shard
// rank and the global lengths).
//
// Design: persistent 2-CTA clusters (one CTA per SM, 192 threads each):
//   warp 0      TMA producer: the 64 rope dims of the query rows once per
//               segment; KV tiles of 64 local rows x 64 dims ("chunks", 8 KB,
//               128-byte swizzle) into a ring of ~22 chunk slots.  Each chunk is
//               fetched once and multicast into both CTAs of the cluster.
//   warp 1      tcgen05 issuer (one thread) and TMEM owner.
//   warps 2-5   load the 512 c_K dims of the query rows into TMEM once per
//               segment, then softmax (one query row per thread) and epilogue.
// A cluster handles a group of at most 96 query rows.  Both CTAs compute the
// same S and P; CTA r keeps value dims [256 r, 256 r + 256).  TMEM per CTA:
// O^T (2 x 96 columns), one S tile (64) and the query's c_K part as the MMA A
// operand (256 columns).  Per tile j:
//   S_j   = Q K_j^T            M=128 rows (A: TMEM for dims 0-511, smem for the
//                              64 rope dims), N=64 KV rows, K=576        -> TMEM fp32
//   P_j   = exp2(S_j*scale*log2e - m)      online softmax with lazy rescaling
//   O^T  += V_j^T P_j^T        M=128 value dims (x2), N=rows, K=64 KV rows -> TMEM fp32
// The tile's chunks stay in the ring from the QK product to the PV product
// (V = the first 512 dims of the same rows), so every KV byte crosses HBM once
// and reaches each SM's shared memory once.  O is kept transposed (dims on
// TMEM lanes) so the accumulator needs only 2 columns per query row per CTA.
//
// Work split (stream-K): units are (request, shard); unit u has T_u tiles.  The
// concatenation of all units' tiles is cut into V equal ranges, one per cluster
// (per row group).  A unit inside one range is written directly; a unit cut by
// range boundaries leaves normalised pieces (o, lse in base 2) in the workspace
// which a second kernel merges with the same LSE rule.  A tiny kernel run first
// writes the tile prefix sums.
#include <cudaTypedefs.h>

#include <mutex>

#include "dcp_internal.cuh"
#include "sm100_ptx.cuh"

using namespace dcp;
using namespace dcp::sm100;

namespace {

constexpr int kTile = 64;          // KV rows per tile
constexpr int kChunkDims = 64;     // dims per chunk (one 128-byte swizzle row)
constexpr int kChunkBytes = kTile * 128;
constexpr int kKSlots = 8;         // main-ring uses per tile: chunks 0-7 (the value dims); pairs start on even slots
constexpr int kMaxSlots = 28;
constexpr int kRopeSlots = 3;      // separate small ring for chunk 8 (the 64 rope dims)
constexpr int kTileBars = 4;       // per-tile "all chunks landed" barriers (> ring depth in tiles)
constexpr int kQTmemCol = 256;     // TMEM columns [256, 512): query dims 0-511 as bf16 pairs
constexpr int kThreads = 224;     // 7 warps: 2 producers, 1 MMA issuer, 4 softmax/epilogue
constexpr int kProducerWarpB = 6;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256
constexpr int kMaxGroupRows = 96;

struct TcArgs {
  Layout L;
  int32_t shard_begin, n_held;
  int32_t B, q_len, H, R_total;  // R_total = q_len * H
  int32_t Rg, ngroups, V;        // rows per group, groups, stream-K ranges
  int32_t nslot;
  int32_t nsbuf;                 // S tiles in TMEM (1 or 2)
  int32_t box_rows;              // KV TMA box height = min(P, 64)
  int64_t pool_rows, pool_pages;
  const int32_t* bt;
  int64_t bt_stride, max_pages;
  const int64_t* seq_lens;
  float scale_log2;
  int32_t base2;
  void* o_part;
  int32_t o_bf16;
  float* lse_part;
  const __nv_bfloat16* q;     // [B * R_total][576]
  const int32_t* tile_start;  // [U + 1]
  float* piece_o;             // [2V][R_total][512]
  float* piece_lse;           // [2V][R_total]
  int32_t* status;
};

struct SmemLayout {
  uint32_t q, ring, rope, p, alpha, inv, vote, bars, misc, total;
};

__host__ __device__ inline SmemLayout smem_layout(int Rg, int nslot) {
  SmemLayout s;
  s.q = 0;                          // rope dims of the query rows: [Rg][64] bf16
  s.ring = Rg * 128;
  s.rope = s.ring + nslot * kChunkBytes;
  s.p = s.rope + kRopeSlots * kChunkBytes;
  s.alpha = s.p + 2 * Rg * 128;
  s.inv = s.alpha + 2 * 128 * 4;
  s.vote = s.inv + 2 * 128 * 4;
  s.bars = s.vote + 64;
  s.misc = s.bars + (2 * kMaxSlots + 2 * kRopeSlots + kTileBars + 16) * 8;
  s.total = s.misc + 64;
  return s;
}

enum Bar { kQFull = 0, kQEmpty, kSFull0, kSFull1, kSFree0, kSFree1, kPFull0, kPFull1, kPFree0, kPFree1, kOFree,
           kGroup, kNumFixedBars };

__device__ inline int64_t unit_nvis_max(const TcArgs& a, int b, int rs, bool* bad) {
  const int64_t S = a.seq_lens[b];
  if (S < a.q_len) {
    *bad = true;
    return 0;
  }
  return count_of(a.shard_begin + rs, S, a.L);
}

// ---------------------------------------------------------------------------- planner
__global__ void __launch_bounds__(1024) plan_kernel(TcArgs a, int32_t* tile_start, int32_t U) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int32_t base = 0; base < U; base += 1024) {
    const int32_t u = base + threadIdx.x;
    int32_t t = 0;
    if (u < U) {
      bool bad = false;
      const int b = u / a.n_held, rs = u % a.n_held;
      const int64_t n = unit_nvis_max(a, b, rs, &bad);
      if (bad && rs == 0) flag(a.status, DCP_STATUS_BAD_LENGTH);
      t = (int32_t)((n + kTile - 1) / kTile);
    }
    // block-wide inclusive scan
    int32_t x = t;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, x, s);
      if (lane >= s) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
      int32_t ws = warp_sums[lane];
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, ws, s);
        if (lane >= s) ws += y;
      }
      warp_sums[lane] = ws;
    }
    __syncthreads();
    const int32_t incl = x + (w > 0 ? warp_sums[w - 1] : 0) + carry;
    if (u < U) tile_start[u] = incl - t;
    __syncthreads();
    if (threadIdx.x == 1023) carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_start[U] = carry;
}

// ---------------------------------------------------------------------------- segments
// A CTA's range [lo, hi) of the global tile sequence, visited unit by unit.
struct SegIter {
  const int32_t* start;
  int32_t U;
  int64_t lo, hi;
  int32_t u;

  __device__ void init(const int32_t* st, int32_t nunits, int64_t lo_, int64_t hi_) {
    start = st; U = nunits; lo = lo_; hi = hi_;
    // largest u with start[u] <= lo
    int32_t l = 0, h = U;  // start[U] = total > lo when lo < hi
    while (h - l > 1) {
      const int32_t m = (l + h) >> 1;
      if (start[m] <= lo) l = m; else h = m;
    }
    u = l;
  }
  // next segment: unit, first tile (within the unit), tile count, whole-unit flag, piece slot
  __device__ bool next(int32_t* unit, int32_t* t0, int32_t* nt, bool* whole, int* kslot) {
    while (u < U) {
      const int64_t s = start[u], e = start[u + 1];
      if (s >= hi) return false;
      const int64_t a = s > lo ? s : lo, b = e < hi ? e : hi;
      const int32_t cur = u++;
      if (a < b) {
        *unit = cur;
        *t0 = (int32_t)(a - s);
        *nt = (int32_t)(b - a);
        *whole = (a == s) && (b == e);
        *kslot = (a == lo) ? 0 : 1;
        return true;
      }
    }
    return false;
  }
};

__device__ inline int64_t range_lo(int64_t T, int v, int V) { return (T * v) / V; }

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2^-22,
// 2^-inf = +0); the result is rounded to bf16 for the PV product anyway.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------- main kernel
// A 2-CTA cluster per work range.  Both CTAs compute the same S and P for the
// group's rows; CTA `rank` accumulates value dims [256 rank, 256 rank + 256)
// (value chunks 4 rank .. 4 rank + 3).  Every KV chunk is fetched once and
// multicast into both CTAs' rings (rank 0 issues the even chunks, rank 1 the odd
// ones); a slot is refilled only when both CTAs have released it.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv,
                      TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout sl = smem_layout(a.Rg, a.nslot);
  unsigned char* qr_s = smem + sl.q;
  unsigned char* ring = smem + sl.ring;
  unsigned char* p_s = smem + sl.p;
  float* alpha_s = reinterpret_cast<float*>(smem + sl.alpha);              // [2][128]
  float* inv_s = reinterpret_cast<float*>(smem + sl.inv);                  // [2][128]
  volatile int* vote_s = reinterpret_cast<volatile int*>(smem + sl.vote);  // [2][4]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bars);
  uint64_t* empty = bars + kNumFixedBars;
  uint64_t* rempty = empty + kMaxSlots;  // rope ring releases
  uint64_t* tfull = rempty + kRopeSlots;  // all 9 chunks of a tile landed in this CTA
  unsigned char* rope = smem + sl.rope;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + sl.misc);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + sl.misc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x >> 1;  // cluster index
  const int v = cid / a.ngroups;
  const int g = cid % a.ngroups;
  const int Rg = a.Rg;
  const int nslot = a.nslot;
  const int nsbuf = a.nsbuf;
  const int32_t U = a.B * a.n_held;
  constexpr uint16_t kBoth = 0x3;

  if (tid == 0) {
    *abort_s = 0;
    for (int i = 0; i < kNumFixedBars; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[kQFull], 5);   // producer (rope TMA bytes) + 4 warps storing Q into TMEM
    mbar_init(&bars[kSFree0], 4);
    mbar_init(&bars[kSFree1], 4);
    mbar_init(&bars[kPFull0], 4);
    mbar_init(&bars[kPFull1], 4);
    mbar_init(&bars[kOFree], 4);
    mbar_init(&bars[kGroup], 4);
    for (int i = 0; i < nslot; ++i) mbar_init(&empty[i], 2);  // released by both CTAs' MMA issuers
    for (int i = 0; i < kRopeSlots; ++i) mbar_init(&rempty[i], 2);
    for (int i = 0; i < kTileBars; ++i) mbar_init(&tfull[i], 2);  // one arrive (with its bytes) per producer
    fence_barrier_init();
  }
  // rows of a page past a request's length are read with zero weight: start from finite zeros
  for (int i = tid; i < (nslot + kRopeSlots) * kChunkBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs exist before any multicast copy or remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;

  const int64_t T = a.tile_start[U];
  const int64_t lo = range_lo(T, v, a.V), hi = range_lo(T, v + 1, a.V);
  const uint32_t ntiles_cta = (uint32_t)(hi - lo);

  if (warp == 0 || warp == kProducerWarpB) {
    // ------------------------------------------------------------------ producers
    // Two producer threads split each tile's ring uses by parity (producer pp
    // handles chunks k = pp, pp + 2, ...), halving the per-use barrier/TMA
    // latency chain; slot parity equals use parity, so each owns half the slots.
    const int pp = warp == 0 ? 0 : 1;
    if (lane == 0 && lo < hi) {
      prefetch_tmap(&tmap_q);
      prefetch_tmap(&tmap_kv);
      SegIter it;
      it.init(a.tile_start, U, lo, hi);
      int32_t u, t0, nt, kslot;
      bool whole;
      uint32_t tile_base = 0;  // first ring use of the current tile (kKSlots per tile)
      int seg = 0;
      bool ok = true;
      // page ids are fetched one tile ahead (raw loads consumed a tile later)
      struct Boxes {
        int32_t y[8];
        uint32_t bytes;
      };
      const int nbox = kTile / a.box_rows;
      auto box_y = [](const Boxes& bx, int q) -> int32_t {  // register-resident select (no local memory)
        int32_t y = bx.y[0];
#pragma unroll
        for (int i = 1; i < 8; ++i)
          if (q == i) y = bx.y[i];
        return y;
      };
      auto fetch_pages = [&](int b, int64_t nvis, int32_t tile, int32_t (&pg)[8]) {
        const int64_t rho0 = (int64_t)tile * kTile;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          pg[q] = -2;  // not needed
          const int64_t rho = rho0 + (int64_t)q * a.box_rows;
          if (q < nbox && rho < nvis) {
            const int64_t pidx = rho / a.L.P;
            pg[q] = pidx < a.max_pages ? __ldg(a.bt + (int64_t)b * a.bt_stride + pidx) : -1;
          }
        }
      };
      auto make_boxes = [&](int rs, int32_t tile, const int32_t (&pg)[8], Boxes& bx) {
        const int64_t rho0 = (int64_t)tile * kTile;
        bx.bytes = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          bx.y[q] = -1;
          if (pg[q] == -2) continue;
          if (pg[q] < 0 || pg[q] >= a.pool_pages) {
            if (rank == 0) flag(a.status, DCP_STATUS_BAD_PAGE_ID);
            continue;
          }
          const int64_t rho = rho0 + (int64_t)q * a.box_rows;
          bx.y[q] = (int32_t)((int64_t)rs * a.pool_rows + (int64_t)pg[q] * a.L.P + rho % a.L.P);
          bx.bytes += a.box_rows * 128;
        }
      };
      // one chunk (all its boxes) into `dst`, completing on `bar`, multicast to both CTAs
      auto issue_chunk = [&](const Boxes& bx, unsigned char* dst, uint64_t* bar, int k) {
        // exactly as many TMA instructions as boxes: predicated-off copies in an
        // unrolled loop still cost the producer issue time
        if (nbox == 1) {
          if (bx.y[0] >= 0) tma_load_2d_multicast(dst, &tmap_kv, bar, k * kChunkDims, bx.y[0], kBoth);
        } else {
          for (int q = 0; q < nbox; ++q) {
            const int32_t y = box_y(bx, q);
            if (y >= 0) tma_load_2d_multicast(dst + q * a.box_rows * 128, &tmap_kv, bar, k * kChunkDims, y, kBoth);
          }
        }
      };
      uint32_t rope_use = 0, tile_idx = 0;
      // Every chunk of a tile completes on the tile's barrier tfull[j % kTileBars]
      // (both producers arrive once with the bytes of their chunks, whichever CTA
      // copies them), so the MMA issuer waits once per tile and issues the whole
      // QK product back to back.
      auto load_tile = [&](const Boxes& bx) -> bool {
        uint64_t* tb = &tfull[tile_idx % kTileBars];
        uint32_t slots[4];
        int n = 0;
        for (int k = pp; k < kKSlots; k += 2) {
          const uint32_t use = tile_base + k;
          const uint32_t slot = use % nslot;
          if (!mbar_wait(&empty[slot], ((use / nslot) & 1) ^ 1, abort_s)) return false;
          slots[n++] = slot;
        }
        uint32_t rslot = 0;
        if (pp == 0) {
          rslot = rope_use % kRopeSlots;
          if (!mbar_wait(&rempty[rslot], ((rope_use / kRopeSlots) & 1) ^ 1, abort_s)) return false;
          ++rope_use;
        }
        mbar_arrive_expect_tx(tb, bx.bytes * (pp == 0 ? 5 : 4));
        if ((int)rank == pp) {  // this CTA copies the chunks of its parity (rank 0 also the rope chunk)
          for (int i = 0; i < n; ++i) issue_chunk(bx, ring + slots[i] * kChunkBytes, tb, pp + 2 * i);
          if (pp == 0) issue_chunk(bx, rope + rslot * kChunkBytes, tb, 8);
        }
        tile_base += kKSlots;
        ++tile_idx;
        return true;
      };
      while (ok && it.next(&u, &t0, &nt, &whole, &kslot)) {
        const int b = u / a.n_held, rs = u % a.n_held;
        bool bad = false;
        const int64_t nvis = unit_nvis_max(a, b, rs, &bad);
        int32_t pg_next[8];
        fetch_pages(b, nvis, t0, pg_next);
        if (pp == 0) {
          if (!mbar_wait(&bars[kQEmpty], (seg & 1) ^ 1, abort_s)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars[kQFull], Rg * 128);
          tma_load_2d(qr_s, &tmap_q, &bars[kQFull], 8 * kChunkDims, b * a.R_total + g * Rg);
        }
        ++seg;
        Boxes cur;
        make_boxes(rs, t0, pg_next, cur);
        for (int jj = 0; jj < nt && ok; ++jj) {
          if (jj + 1 < nt) fetch_pages(b, nvis, t0 + jj + 1, pg_next);
          ok = load_tile(cur);
          if (jj + 1 < nt) make_boxes(rs, t0 + jj + 1, pg_next, cur);
        }
      }
      // Drain: every release addressed to this CTA's ring (including the peer's
      // remote ones) lands before the cluster may retire.  Bounded; skipped
      // after an abort.
      if (ok) {
        const uint32_t total = ntiles_cta * kKSlots;
        for (uint32_t s = pp; s < (uint32_t)nslot && s < total; s += 2) {
          const uint32_t last = s + ((total - 1 - s) / nslot) * nslot;  // last use of slot s
          if (!mbar_wait(&empty[s], (last / nslot) & 1, abort_s)) break;
        }
        if (pp == 0) {
          for (uint32_t s = 0; s < (uint32_t)kRopeSlots && s < ntiles_cta; ++s) {
            const uint32_t last = s + ((ntiles_cta - 1 - s) / kRopeSlots) * kRopeSlots;
            if (!mbar_wait(&rempty[s], (last / kRopeSlots) & 1, abort_s)) break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Event-driven single thread: QK chunks are issued as their data lands and
    // each PV product as soon as its P tile is ready.
    if (lane == 0 && lo < hi) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, kTile, 0, 0);
      const uint32_t idesc_pv = idesc_bf16_f32(128, Rg, 1, 0);
      const uint64_t kdesc0 = sw128_desc(smem_u32(ring), 16, 1024);
      const uint64_t vdesc0 = sw128_desc(smem_u32(ring), kChunkBytes, 1024);
      const uint64_t qrdesc0 = sw128_desc(smem_u32(qr_s), 16, 1024);
      const uint64_t pdesc0 = sw128_desc(smem_u32(p_s), 16, 1024);
      const int my_lo = 4 * (int)rank;  // value chunks this CTA keeps for its PV product
      const uint64_t rdesc0 = sw128_desc(smem_u32(rope), 16, 1024);
      // QK product of chunk k (< 8: value dims from the main ring; 8: rope dims)
      auto issue_qk_chunk = [&](uint32_t j, int k, uint32_t slot) {
        const uint32_t d = tmem + 2 * Rg + kTile * (j % nsbuf);
        if (k < 8) {
          const uint64_t kd = kdesc0 + ((slot * kChunkBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(d, tmem + kQTmemCol + k * 32 + kk * 8, kd + kk * 2, idesc_qk, (k | kk) != 0);
          if (k < my_lo || k >= my_lo + 4) mma_commit_multicast(&empty[slot], kBoth);  // not one of my V chunks
        } else {
          const uint64_t kd = rdesc0 + ((slot * kChunkBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(d, qrdesc0 + kk * 2, kd + kk * 2, idesc_qk, 1);
          mma_commit_multicast(&rempty[slot], kBoth);
        }
      };
      auto issue_pv = [&](uint32_t j, bool first) {
        const int pb = j & 1;
        const uint64_t pd = pdesc0 + ((pb * Rg * 128) >> 4);
        const uint32_t base = j * kKSlots + my_lo;
        for (int t = 0; t < 2; ++t) {
          const uint32_t slot = (base + 2 * t) % nslot;  // even: the pair (2t, 2t+1) is contiguous
          const uint64_t vd = vdesc0 + ((slot * kChunkBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(tmem + t * Rg, vd + kk * (2048 >> 4), pd + kk * 2, idesc_pv, !(first && kk == 0));
          mma_commit_multicast(&empty[slot], kBoth);
          mma_commit_multicast(&empty[slot + 1], kBoth);
        }
        mma_commit(&bars[kPFree0 + pb]);
      };
      SegIter itq;
      itq.init(a.tile_start, U, lo, hi);
      int32_t uq, t0q, ntq, ksq;
      bool wq;
      bool q_has = itq.next(&uq, &t0q, &ntq, &wq, &ksq);
      int q_seg = 0, q_jj = 0;
      bool q_seg_ready = false, q_tile_ready = false;
      uint32_t jq = 0;
      SegIter itp;
      itp.init(a.tile_start, U, lo, hi);
      int32_t up, t0p, ntp, ksp;
      bool wp;
      bool p_has = itp.next(&up, &t0p, &ntp, &wp, &ksp);
      int p_seg = 0, p_jj = 0;
      uint32_t jp = 0;
      uint64_t idle_since = 0;
      uint32_t idle_polls = 0;
      uint32_t m_slot = 0, r_slot = 0;  // next main-ring and rope-ring slots the QK cursor reads
      while (q_has || p_has) {
        bool progress = false;
        if (p_has && jp < jq) {
          bool ready = mbar_test(&bars[kPFull0 + (jp & 1)], (jp >> 1) & 1);
          if (ready && p_jj == 0 && p_seg >= 1) ready = mbar_test(&bars[kOFree], (p_seg - 1) & 1);
          if (ready) {
            tc_fence_after();
            issue_pv(jp, p_jj == 0);
            ++jp;
            if (++p_jj == ntp) {
              ++p_seg;
              p_jj = 0;
              p_has = itp.next(&up, &t0p, &ntp, &wp, &ksp);
            }
            progress = true;
          }
        }
        if (q_has) {
          if (!q_seg_ready && mbar_test(&bars[kQFull], q_seg & 1)) {
            q_seg_ready = true;
            progress = true;
          }
          if (q_seg_ready && !q_tile_ready &&
              mbar_test(&bars[kSFree0 + (jq % nsbuf)], ((jq / nsbuf) & 1) ^ 1)) {
            q_tile_ready = true;
            progress = true;
          }
          if (q_tile_ready && mbar_test(&tfull[jq % kTileBars], (jq / kTileBars) & 1)) {
            // all 9 chunks of tile jq have landed: the whole QK product back to back
            tc_fence_after();
            for (int k = 0; k < kKSlots; ++k) {
              issue_qk_chunk(jq, k, m_slot);
              if (++m_slot == (uint32_t)nslot) m_slot = 0;
            }
            issue_qk_chunk(jq, kKSlots, r_slot);
            if (++r_slot == (uint32_t)kRopeSlots) r_slot = 0;
            mma_commit(&bars[kSFull0 + (jq % nsbuf)]);
            if (q_jj == ntq - 1) mma_commit(&bars[kQEmpty]);
            ++jq;
            q_tile_ready = false;
            if (++q_jj == ntq) {
              ++q_seg;
              q_jj = 0;
              q_seg_ready = false;
              q_has = itq.next(&uq, &t0q, &ntq, &wq, &ksq);
            }
            progress = true;
          }
        }
        if (progress) {
          idle_since = 0;
          idle_polls = 0;
        } else if ((++idle_polls & 31) == 0) {  // look at the clock every 32 idle polls
          if (*abort_s) break;
          const uint64_t now = globaltimer();
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > kWaitLimitNs) {
            *abort_s = 1;
            break;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ Q load, softmax, epilogue
    // Waits are polled by one lane per warp and broadcast; the four warps meet
    // only through bounded mbarriers, so a timeout drains every thread.
    const int c = 32 * (warp & 3) + lane;        // TMEM lane: query row (S, Q) / value dim (O^T)
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    if (lo < hi) {
      auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
        int r = 1;
        if (lane == 0) r = mbar_wait(bar, parity, abort_s) ? 1 : 0;
        r = __shfl_sync(0xffffffffu, r, 0);
        return r != 0;
      };
      uint32_t gphase = 0;  // kGroup phases passed
      auto group_sync = [&](bool flag_in, bool* any) -> bool {
        const bool wany = __any_sync(0xffffffffu, flag_in);
        if (lane == 0) vote_s[(gphase & 1) * 4 + (warp & 3)] = wany ? 1 : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kGroup]);
        if (!wwait(&bars[kGroup], gphase & 1)) return false;
        const int base = (gphase & 1) * 4;
        *any = vote_s[base] | vote_s[base + 1] | vote_s[base + 2] | vote_s[base + 3];
        ++gphase;
        return true;
      };
      SegIter it;
      it.init(a.tile_start, U, lo, hi);
      int32_t u, t0, nt, kslot;
      bool whole;
      uint32_t jglob = 0;
      int seg = 0;
      bool ok = true;
      // PV #k completes phase k/2 of p_free[k % 2]; that barrier cannot run two
      // phases ahead of this wait (its next phase needs P of tile k + 2).
      auto wait_pv = [&](uint32_t k) -> bool { return wwait(&bars[kPFree0 + (k & 1)], (k >> 1) & 1); };
      while (ok && it.next(&u, &t0, &nt, &whole, &kslot)) {
        const int b = u / a.n_held, rs = u % a.n_held;
        const int64_t S = a.seq_lens[b];
        const int grow = g * Rg + c;
        const bool active = c < Rg && grow < a.R_total && S >= a.q_len;
        int64_t nvis = 0;
        if (active) nvis = count_of(a.shard_begin + rs, S - a.q_len + grow / a.H + 1, a.L);
        // ---- query dims 0-511 of this row -> TMEM lane c, columns [256, 512)
        if (!wwait(&bars[kQEmpty], (seg & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        {
          const bool has_row = c < Rg && grow < a.R_total;
          const uint4* src = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.R_total + grow) * kDk);
          for (int i = 0; i < 8; ++i) {
            uint32_t r[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              uint4 w4 = has_row ? __ldg(src + 8 * i + k) : make_uint4(0, 0, 0, 0);
              r[4 * k] = w4.x; r[4 * k + 1] = w4.y; r[4 * k + 2] = w4.z; r[4 * k + 3] = w4.w;
            }
            tmem_st32(tmem + lane_base + kQTmemCol + 32 * i, r);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kQFull]);
        ++seg;
        float m_ref = -INFINITY, l = 0.f;
        for (int jj = 0; jj < nt; ++jj, ++jglob) {
          const int sb = jglob % nsbuf;
          if (!wwait(&bars[kSFull0 + sb], (jglob / nsbuf) & 1)) { ok = false; break; }
          tc_fence_after();
          uint32_t sr[64];
          tmem_ld32(tmem + lane_base + 2 * Rg + kTile * sb, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          tmem_ld32(tmem + lane_base + 2 * Rg + kTile * sb + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kSFree0 + sb]);
          const int64_t rho0 = (int64_t)(t0 + jj) * kTile;
          const int64_t lim = nvis - rho0;  // columns k < lim are visible to this row
          if (lim < kTile) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (k >= lim) sr[k] = __float_as_uint(-INFINITY);
          }
          float mraw = -INFINITY;
#pragma unroll
          for (int k = 0; k < 64; ++k) mraw = fmaxf(mraw, __uint_as_float(sr[k]));
          const float mt = mraw * a.scale_log2;  // scale > 0: the max commutes with the scaling
          bool need = false;
          float alpha = 1.f;
          if (m_ref == -INFINITY) {
            m_ref = mt;  // nothing accumulated yet for this row
          } else if (mt > m_ref + kRescaleThreshold) {
            need = true;
            alpha = exp2f(m_ref - mt);
            m_ref = mt;
          }
          const uint32_t abuf = (gphase & 1) * 128;
          alpha_s[abuf + c] = alpha;
          bool any = false;
          if (!group_sync(need, &any)) { ok = false; break; }
          const int pb = jglob & 1;
          if (!wwait(&bars[kPFree0 + pb], ((jglob >> 1) & 1) ^ 1)) { ok = false; break; }
          if (any) {
            // O^T columns of the rows whose maximum moved are scaled by alpha
            if (!wait_pv(jglob - 1)) { ok = false; break; }
            tc_fence_after();
            for (int t = 0; t < 2; ++t) {
              for (int c0 = 0; c0 < Rg; c0 += 16) {
                uint32_t r[16];
                const uint32_t addr = tmem + lane_base + t * Rg + c0;
                tmem_ld16(addr, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha_s[abuf + c0 + i]);
                tmem_st16(addr, r);
              }
            }
            tmem_st_wait();
            l *= alpha;
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          const float cs = a.scale_log2;
          float psum = 0.f;
          uint32_t pk[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * k]), cs, -m_use));
            const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * k + 1]), cs, -m_use));
            psum += p0 + p1;
            __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
            pk[k] = *reinterpret_cast<uint32_t*>(&h);
          }
          l += psum;
          if (c < Rg) {
            // row c of the K-major, 128B-swizzled P tile: 8 x 16-byte pieces
            unsigned char* row = p_s + pb * Rg * 128 + (c >> 3) * 1024 + (c & 7) * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              uint4 w4 = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
              *reinterpret_cast<uint4*>(row + ((q ^ (c & 7)) << 4)) = w4;
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kPFull0 + pb]);
        }
        if (!ok) break;
        // ---------------- epilogue: O^T (my dims x rows) / l -> o, lse
        if (!wait_pv(jglob - 1)) { ok = false; break; }
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const uint32_t ibuf = (gphase & 1) * 128;
        inv_s[ibuf + c] = inv;
        const float lse2 = l > 0.f ? m_ref + log2f(l) : -INFINITY;
        bool dummy;
        if (!group_sync(false, &dummy)) { ok = false; break; }
        const int R_here = min(Rg, a.R_total - g * Rg);
        const int64_t out_row0 = ((int64_t)rs * a.B + b) * a.R_total + g * Rg;
        const int64_t piece = (int64_t)(2 * v + kslot) * a.R_total + g * Rg;
        for (int t = 0; t < 2; ++t) {
          for (int c0 = 0; c0 < Rg; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + lane_base + t * Rg + c0, r);
            tmem_ld_wait();
            const int dim = 256 * (int)rank + t * 128 + c;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int row = c0 + i;
              if (row < R_here) {
                const float val = __uint_as_float(r[i]) * inv_s[ibuf + row];
                if (whole) {
                  if (a.o_bf16)
                    static_cast<__nv_bfloat16*>(a.o_part)[(out_row0 + row) * kDv + dim] = __float2bfloat16_rn(val);
                  else
                    static_cast<float*>(a.o_part)[(out_row0 + row) * kDv + dim] = val;
                } else {
                  a.piece_o[(piece + row) * kDv + dim] = val;
                }
              }
            }
          }
        }
        if (c < R_here && rank == 0) {
          if (whole)
            a.lse_part[out_row0 + c] = a.base2 ? lse2 : lse2 * kLn2;
          else
            a.piece_lse[piece + c] = lse2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kOFree]);
      }
    }
  }

  if (*abort_s && tid == 0) flag(a.status, DCP_STATUS_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  // The peer may still have copies or arrivals addressed to this CTA's shared
  // memory; retire the pair together.  After an abort, allow in-flight tensor
  // core commits (microseconds) to land first.
  if (*abort_s) __nanosleep(100000);
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------- fixup
// Writes empty units (o = 0, lse = -inf) and merges the pieces of units cut by
// range boundaries.  One block per unit.
__global__ void __launch_bounds__(256) fixup_kernel(TcArgs a) {
  const int32_t U = a.B * a.n_held;
  const int32_t u = blockIdx.x;
  if (u >= U) return;
  const int b = u / a.n_held, rs = u % a.n_held;
  const int64_t s = a.tile_start[u], e = a.tile_start[u + 1];
  const int64_t T = a.tile_start[U];
  const int64_t out_row0 = ((int64_t)rs * a.B + b) * a.R_total;
  const int64_t nelem = (int64_t)a.R_total * kDv;
  if (s == e) {
    for (int64_t i = threadIdx.x; i < nelem; i += blockDim.x) {
      if (a.o_bf16) static_cast<__nv_bfloat16*>(a.o_part)[out_row0 * kDv + i] = __float2bfloat16_rn(0.f);
      else static_cast<float*>(a.o_part)[out_row0 * kDv + i] = 0.f;
    }
    for (int i = threadIdx.x; i < a.R_total; i += blockDim.x) a.lse_part[out_row0 + i] = -INFINITY;
    return;
  }
  const int V = a.V;
  auto part_of = [&](int64_t x) {  // range containing tile x
    int vv = (int)((x * V) / T);
    while (vv + 1 < V && range_lo(T, vv + 1, V) <= x) ++vv;
    while (vv > 0 && range_lo(T, vv, V) > x) --vv;
    return vv;
  };
  const int v0 = part_of(s), v1 = part_of(e - 1);
  if (v0 == v1) return;  // written whole by the main kernel
  // each thread handles (row, 4 dims) items
  for (int64_t item = threadIdx.x; item < (int64_t)a.R_total * (kDv / 4); item += blockDim.x) {
    const int row = (int)(item / (kDv / 4));
    const int d4 = (int)(item % (kDv / 4)) * 4;
    float m = -INFINITY;
    for (int vv = v0; vv <= v1; ++vv) {
      if (range_lo(T, vv, V) == range_lo(T, vv + 1, V)) continue;  // empty range: no piece
      const int k = range_lo(T, vv, V) >= s ? 0 : 1;
      m = fmaxf(m, a.piece_lse[(int64_t)(2 * vv + k) * a.R_total + row]);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int vv = v0; vv <= v1; ++vv) {
        if (range_lo(T, vv, V) == range_lo(T, vv + 1, V)) continue;
        const int k = range_lo(T, vv, V) >= s ? 0 : 1;
        const int64_t pr = (int64_t)(2 * vv + k) * a.R_total + row;
        const float lv = a.piece_lse[pr];
        if (lv == -INFINITY) continue;
        const float w = exp2f(lv - m);
        wsum += w;
        const float4 o4 = *reinterpret_cast<const float4*>(a.piece_o + pr * kDv + d4);
        acc[0] = fmaf(w, o4.x, acc[0]);
        acc[1] = fmaf(w, o4.y, acc[1]);
        acc[2] = fmaf(w, o4.z, acc[2]);
        acc[3] = fmaf(w, o4.w, acc[3]);
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int64_t o_idx = (out_row0 + row) * kDv + d4;
    for (int i = 0; i < 4; ++i) {
      if (a.o_bf16) static_cast<__nv_bfloat16*>(a.o_part)[o_idx + i] = __float2bfloat16_rn(acc[i] * inv);
      else static_cast<float*>(a.o_part)[o_idx + i] = acc[i] * inv;
    }
    if (d4 == 0) {
      const float lse2 = wsum > 0.f ? m + log2f(wsum) : -INFINITY;
      a.lse_part[out_row0 + row] = a.base2 ? lse2 : lse2 * kLn2;
    }
  }
}

// ---------------------------------------------------------------------------- host side
struct Plan {
  int Rg, ngroups, V, nslot, nsbuf, box_rows;
  size_t smem;
  size_t ws_start_bytes, ws_piece_o_bytes, ws_piece_lse_bytes, ws_total;
};

int sm_count_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int max_active_clusters(size_t smem) {
  static size_t cached_smem = 0;
  static int cached = -1, cached_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cached >= 0 && cached_smem == smem && cached_dev == dev) return cached;
  if (cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 512, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, partial_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached = n;
  cached_smem = smem;
  cached_dev = dev;
  return n;
}

bool make_plan(const dcp_layout_t* layout, int n_held, int B, int q_len, int H, Plan* p) {
  const int R_total = q_len * H;
  p->ngroups = (R_total + kMaxGroupRows - 1) / kMaxGroupRows;
  const int per = (R_total + p->ngroups - 1) / p->ngroups;
  p->Rg = ((per + 15) / 16) * 16;
  const int sms = sm_count_current();
  if (sms <= 0) return false;
  p->V = (sms / 2) / p->ngroups;  // ranges: one 2-CTA cluster per (range, row group)
  if (p->V < 1) p->V = 1;
  const SmemLayout base = smem_layout(p->Rg, 0);
  const size_t budget = 232448 - 1024;  // 227 KB minus alignment slack
  int nslot = (int)((budget - base.total) / kChunkBytes);
  nslot &= ~1;
  if (nslot > kMaxSlots) nslot = kMaxSlots;
  p->nslot = nslot;
  p->nsbuf = (2 * p->Rg + 2 * kTile <= kQTmemCol) ? 2 : 1;
  p->smem = smem_layout(p->Rg, nslot).total + 1024;
  // clusters that can be resident at once (both CTAs of a cluster share a GPC)
  const int clusters = max_active_clusters(p->smem);
  if (clusters > 0) {
    p->V = clusters / p->ngroups;
    if (p->V < 1) p->V = 1;
  }
  const int P = layout->page_size;
  p->box_rows = P >= kTile ? kTile : P;
  const int64_t U = (int64_t)B * n_held;
  p->ws_start_bytes = align256((size_t)(U + 1) * 4);
  p->ws_piece_o_bytes = align256((size_t)2 * p->V * R_total * kDv * 4);
  p->ws_piece_lse_bytes = align256((size_t)2 * p->V * R_total * 4);
  p->ws_total = p->ws_start_bytes + p->ws_piece_o_bytes + p->ws_piece_lse_bytes;
  return nslot >= 2 * kKSlots;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 [rows, 576] row-major, 128-byte swizzled boxes of [box_rows, 64]
bool make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDk, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDk * 2};
  cuuint32_t box[2] = {(cuuint32_t)kChunkDims, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool page_size_ok(int P) { return P >= 8 && P % 8 == 0 && (P % kTile == 0 || kTile % P == 0); }

}  // namespace

extern "C" size_t dcp_mla_decode_workspace_size(const dcp_layout_t* layout, int32_t shard_begin,
                                                int32_t shard_end, int32_t B, int32_t q_len, int32_t H) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end ||
      B < 1 || q_len < 1 || H < 1 || (int64_t)q_len * H > 1024)
    return 0;
  Plan p;
  if (!make_plan(layout, shard_end - shard_begin, B, q_len, H, &p)) return 0;
  return p.ws_total;
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
  if (!page_size_ok(layout->page_size)) return DCP_ERR_UNSUPPORTED;
  const int n_held = shard_end - shard_begin;
  const int64_t pool_rows = pool_pages * layout->page_size;
  if ((int64_t)n_held * pool_rows >= INT32_MAX || (int64_t)B * q_len * H >= INT32_MAX ||
      (int64_t)B * n_held >= INT32_MAX / 2)
    return DCP_ERR_UNSUPPORTED;
  Plan p;
  if (!make_plan(layout, n_held, B, q_len, H, &p)) return DCP_ERR_CUDA;
  if (!workspace || workspace_bytes < p.ws_total) return DCP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return DCP_ERR_INVALID;

  CUtensorMap tq, tkv;
  if (!make_tmap(&tq, q, (uint64_t)B * q_len * H, (uint32_t)p.Rg)) return DCP_ERR_CUDA;
  if (!make_tmap(&tkv, arena, (uint64_t)n_held * pool_rows, (uint32_t)p.box_rows)) return DCP_ERR_CUDA;

  static size_t smem_set = 0;
  if (smem_set < p.smem) {
    if (cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
        cudaSuccess)
      return DCP_ERR_CUDA;
    smem_set = p.smem;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  TcArgs a;
  a.L = to_layout(layout);
  a.shard_begin = shard_begin;
  a.n_held = n_held;
  a.B = B; a.q_len = q_len; a.H = H; a.R_total = q_len * H;
  a.Rg = p.Rg; a.ngroups = p.ngroups; a.V = p.V; a.nslot = p.nslot; a.nsbuf = p.nsbuf; a.box_rows = p.box_rows;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.pool_rows = pool_rows; a.pool_pages = pool_pages;
  a.bt = block_table; a.bt_stride = bt_stride; a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.scale_log2 = scale * kLog2e;
  a.base2 = lse_base == DCP_LSE_BASE_2;
  a.o_part = o_part; a.o_bf16 = o_part_dtype == DCP_BF16;
  a.lse_part = lse_part;
  a.tile_start = reinterpret_cast<const int32_t*>(ws);
  a.piece_o = reinterpret_cast<float*>(ws + p.ws_start_bytes);
  a.piece_lse = reinterpret_cast<float*>(ws + p.ws_start_bytes + p.ws_piece_o_bytes);
  a.status = status;
  cudaStream_t st = as_stream(stream);
  const int32_t U = B * n_held;
  plan_kernel<<<1, 1024, 0, st>>>(a, reinterpret_cast<int32_t*>(ws), U);
  partial_tc_kernel<<<2 * p.V * p.ngroups, kThreads, p.smem, st>>>(tq, tkv, a);
  fixup_kernel<<<U, 256, 0, st>>>(a);
  return launch_status(3);
}

// ---------------------------------------------------------------------------- allocation-free variant
// Some callers cannot hand the library a workspace: a serving process that has
// given every free byte of HBM to its KV pool and forbids further device
// allocations, or a plain C host with no device-memory manager of its own.
// For them the partial decode can run on a scratch area that the library owns:
// a file-scope device array, created when the library is loaded on a device and
// kept until the process exits.
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB per device
__device__ __align__(256) unsigned char g_partial_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_partial_scratch on the current device (looked up once per
// device; in host code the array's name is only a host-side stand-in).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_partial_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" size_t dcp_mla_decode_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" int32_t dcp_mla_decode_partial_static(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                                                 const void* q, int32_t B, int32_t q_len, int32_t H,
                                                 const void* arena, int64_t pool_pages,
                                                 const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                                                 const int64_t* seq_lens, float scale, int32_t lse_base,
                                                 void* o_part, int32_t o_part_dtype, float* lse_part,
                                                 int32_t* status, void* stream) {
  const size_t need = dcp_mla_decode_workspace_size(layout, shard_begin, shard_end, B, q_len, H);
  if (need == 0) return DCP_ERR_INVALID;
  if (need > kStaticScratchBytes) return DCP_ERR_TOO_LARGE;
  void* ws = scratch_address();
  if (!ws) return DCP_ERR_CUDA;
  return dcp_mla_decode_partial(layout, shard_begin, shard_end, q, B, q_len, H, arena, pool_pages, block_table,
                                bt_stride, max_pages, seq_lens, scale, lse_base, o_part, o_part_dtype, lse_part, ws,
                                kStaticScratchBytes, status, stream);
}
