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
// Design: persistent 2-CTA clusters, one CTA per SM, 384 threads each:
//   warps 0-7   softmax and score exchange: warp w serves 16 query rows
//               (two threads per row, 32 keys each); it loads its rows of this
//               CTA's query chunks into TMEM once per segment, ships its rows
//               of each partial score tile to the peer, runs the online
//               softmax and writes its rows of O at a segment end.
//   warp 9      PV issuer (one thread).
//   warp 10     TMA producer: this CTA's share of every KV tile (64 local rows)
//               into a ring of tile slots, an L2 prefetch two tiles ahead, and
//               the query's shared-memory operands once per segment.  The warp
//               fetches block-table entries 32 tiles at a time.
//   warp 11     QK issuer (one thread) and TMEM owner.
// A cluster handles a group of at most 128 query rows.  The 576 key dims are
// split between the two CTAs: CTA r loads value chunks 4r .. 4r + 3 (dims
// [256 r, 256 r + 256), one 3-D box of four 128-byte-swizzled 64 x 64 tiles)
// and rope dims [512 + 32 r, 512 + 32 r + 32) (64-byte swizzle).  Per tile j,
// in each CTA:
//   S_j^r = Q[:, K_r] K_j[:, K_r]^T   M=128 rows, N=64 KV rows, K=288: query
//                                     chunks 4r, 4r+1 from TMEM, chunks 4r+2,
//                                     4r+3 and the rope half from shared
//                                     memory -> TMEM fp32
//   each softmax warp stages its rows of S_j^r in shared memory and one bulk
//   copy ships them to the peer (credited on the peer's mbarrier; two buffers
//   per CTA swap the staging and receiving roles every tile); each CTA forms
//   S_j = S_j^0 + S_j^1 (fp32 addition is commutative, so both CTAs hold the
//   same bits and take the same softmax decisions);
//   P_j   = exp2(S_j*scale*log2e - m)  online softmax with lazy rescaling,
//                                     bf16 pairs in their own TMEM columns
//   O_r  += P_j V_j[:, dims of r]     M=128 rows (A = P from TMEM), N=256,
//                                     K=64 KV rows                   -> TMEM fp32
// Each KV byte crosses HBM once and reaches one SM's shared memory once; the
// tile's chunks stay in the ring from the QK product to the PV product (V = the
// first 512 dims of the same rows).  TMEM per CTA: O (256 columns), two S
// tiles (2 x 64), two P tiles (2 x 32) and two query chunks (64).  An S tile
// is free as soon as every softmax warp has read it, so QK products run up to
// two tiles ahead of the softmax while the exchange is in flight.
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

constexpr int kTile = 64;                     // KV rows per tile
constexpr int kChunkDims = 64;                // dims per chunk (one 128-byte swizzle row)
constexpr int kChunkBytes = kTile * 128;      // 8 KB
constexpr int kOwnChunks = 4;                 // value chunks each CTA loads (256 dims)
constexpr int kRopeHalf = 32;                 // rope dims each CTA loads (64-byte swizzled rows)
constexpr int kRopeHalfBytes = kTile * 64;
constexpr int kRopeOff = kOwnChunks * kChunkBytes;         // rope part inside a tile slot
constexpr int kSlotBytes = kRopeOff + kRopeHalfBytes;      // 36 KB per tile slot
constexpr int kMaxTileSlots = 8;
constexpr int kL2Ahead = 2;                   // tiles between a tile's L2 prefetch and its ring load
constexpr int kFixedBarSlots = 32;            // mbarriers other than the per-slot ones
constexpr int kThreads = 384;                 // 12 warps (roles below)
// Warp roles.  Warp w runs on SM sub-partition w % 4 and reaches TMEM lanes
// [32 (w % 4), 32 (w % 4) + 32): the softmax and sender warps of row quarter q
// are q and 4 + q.  The tensor-core issuer (a polling thread) sits with the
// warps of quarter 3, the quarter a group of up to 96 rows leaves empty, and
// the producer with quarter 2; warps 8 and 9 have no role.
constexpr int kHalfRows = 16;                 // rows served by one softmax warp (two threads per row)
constexpr int kProducerWarp = 10;
constexpr int kMmaWarp = 11;                  // QK issuer and TMEM owner
constexpr int kPvWarp = 9;                    // PV issuer
constexpr int kMaxGroupRows = 128;
constexpr int64_t kMaxQueryRows = 65536;      // q_len * H per request (512 row groups)
constexpr uint32_t kOCol = 0;                 // TMEM columns [0, 256): O, rows on lanes
constexpr uint32_t kSCol = 256;               // [256, 384): two S tiles of 64 fp32 columns
constexpr uint32_t kPCol = 384;               // [384, 448): P of two tiles as bf16 pairs (2 x 32)
constexpr uint32_t kQCol = 448;               // [448, 512): query chunks 4r, 4r + 1 as bf16 pairs
constexpr int kQTmemChunks = 2;               // query chunks 4r + 2, 4r + 3 are read from shared memory
constexpr int kXRowBytes = kTile * 4;         // one row of a partial score tile (fp32)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: P stays <= 256

struct TcArgs {
  Layout L;
  int32_t shard_begin, n_held;
  int32_t B, q_len, H, R_total;  // R_total = q_len * H
  int32_t Rg, ngroups, V;        // rows per group, groups, stream-K ranges
  int32_t nts;                   // tile slots in the ring
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
  uint32_t qc, qr, x, xbuf, ring, rope, bars, misc, total;
};

__host__ __device__ inline uint32_t round1024(uint32_t v) { return (v + 1023u) & ~1023u; }

__host__ __device__ inline SmemLayout smem_layout(int Rg, int nts) {
  SmemLayout s;
  // The M = 128 shared-memory A operands hold the group's Rg rows; the products
  // also read the 128 - Rg rows that follow into TMEM lanes no thread reads
  // back.  Query chunk 4r + 2 is given all 128 rows, zeroed, so its padding
  // rows multiply zeros (less power at the power cap); chunk 4r + 3 and the
  // rope dims are followed by other data, as the ring needs the space.
  s.qc = 0;                                        // query chunks 4r + 2 ([128][64], rows >= Rg zero), 4r + 3 ([Rg][64]), bf16, 128-byte swizzle
  s.qr = (128 + (uint32_t)Rg) * 128;               // query rope dims [32r, 32r + 32): [Rg][32], 64-byte swizzle
  s.x = round1024(s.qr + (uint32_t)Rg * 64);       // two [Rg][64] fp32 buffers: partial scores staged / received
  s.xbuf = round1024((uint32_t)Rg * kXRowBytes);
  s.ring = s.x + 2 * s.xbuf;                       // tile slots: 4 value chunks + this CTA's rope half
  s.rope = s.ring;                                 // (kept for the layout struct; rope lives in the slots)
  s.bars = s.ring + nts * kSlotBytes;
  s.misc = s.bars + (kFixedBarSlots + 2 * kMaxTileSlots) * 8;
  s.total = s.misc + 64;
  return s;
}

enum Bar { kQFull = 0, kQEmpty, kSFull0, kSFull1, kSFree0, kSFree1, kPFull0, kPFull1, kPVDone0, kPVDone1, kOFree,
           kXFull = 11,  // [2 buffers][8 channels]: the peer's partial scores of a channel's rows have landed
           kNumFixedBars = 27 };
static_assert(kNumFixedBars <= kFixedBarSlots, "fixed barriers");

__device__ inline int64_t unit_nvis_max(const TcArgs& a, int b, int rs, bool* bad) {
  const int64_t S = a.seq_lens[b];
  if (S < a.q_len) {
    *bad = true;
    return 0;
  }
  return count_of(a.shard_begin + rs, S, a.L);
}

// ---------------------------------------------------------------------------- planner
// Tile prefix sums of the (request, shard) units, and the rows of units with no
// visible key (an empty shard): o = 0 and lse = -inf, written here because the
// main kernel never visits them.  One block of 1024 threads, 1024 units per pass.
__global__ void __launch_bounds__(1024) plan_kernel(TcArgs a, int32_t* tile_start, int32_t U) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  __shared__ int32_t empty_s[1024];
  __shared__ int32_t n_empty_s;
  if (threadIdx.x == 0) {
    carry = 0;
    n_empty_s = 0;
  }
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
      if (t == 0) empty_s[atomicAdd(&n_empty_s, 1)] = u;  // at most 1024 per pass
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
    // this pass's empty units: every thread writes 16-byte pieces of their rows
    const int n_empty = n_empty_s;
    const int64_t row_bytes = (int64_t)kDv * (a.o_bf16 ? 2 : 4);
    for (int k = 0; k < n_empty; ++k) {
      const int32_t ue = empty_s[k];
      const int64_t row0 = ((int64_t)(ue % a.n_held) * a.B + ue / a.n_held) * a.R_total;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(a.o_part) + row0 * row_bytes);
      for (int64_t i = threadIdx.x; i < a.R_total * row_bytes / 16; i += 1024) dst[i] = make_uint4(0, 0, 0, 0);
      for (int i = threadIdx.x; i < a.R_total; i += 1024) a.lse_part[row0 + i] = -INFINITY;
    }
    __syncthreads();
    if (threadIdx.x == 0) n_empty_s = 0;
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

// Two fp32 values in one 64-bit register pair, for the packed FP32 operations
// of sm_100 (two lanes per instruction; each lane rounds as its scalar form).
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, uint32_t& lo, uint32_t& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2^-22,
// 2^-inf = +0); the result is rounded to bf16 for the PV product anyway.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp-uniform bounded waits.  Fast path: every lane tests the phase once (its
// own acquire) and one vote confirms; otherwise each lane waits with the bounded
// loop and a final vote makes the outcome uniform (false after an abort).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_s, int lane) {
  bool ok = mbar_try_wait(bar, parity);  // every lane: its own acquire
  if (__all_sync(0xffffffffu, ok)) return true;
  if (!ok) ok = mbar_wait(bar, parity, abort_s);
  return __all_sync(0xffffffffu, ok);  // warp-uniform (false after an abort)
}

__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_s, int lane) {
  bool ok = mbar_try_wait_cluster(bar, parity);
  if (__all_sync(0xffffffffu, ok)) return true;
  if (!ok) ok = mbar_wait_cluster(bar, parity, abort_s);
  return __all_sync(0xffffffffu, ok);
}

// O rows of one softmax warp scaled by f (16 lanes from `o_addr`'s lane;
// thread t: row t % 16, columns [128 (t / 16), 128 (t / 16) + 128)).
__device__ __forceinline__ void rescale_rows(uint32_t o_addr, float f) {
#pragma unroll 1
  for (int k = 0; k < 4; ++k) {
    uint32_t r[32];
    tmem_ld16x2_sync<128>(o_addr + 32 * k, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
    tmem_st16x2<128>(o_addr + 32 * k, r);
    tmem_st_wait();  // before the next load reuses r
  }
}

// The same O rows times `inv` -> the output rows (bf16 or fp32) or the fp32
// piece rows; thread t holds dims [d0, d0 + 128) of row r0 + t % 16.  Rows
// [0, rows_here) of the group are written.  Kept out of line: it runs once per
// segment and inlining it cost the tile loop.
//
// fp32 rows go through `stage`, this warp's 16 rows of the score-exchange
// buffer it read the peer's last tile from (4 KB: 64 floats per row, 16-byte
// chunk c of row r at chunk slot c ^ (r % 16), as the exchange lays them out);
// nothing writes those rows again before this warp ships its next tile.  Per 32
// dims, each thread writes its row segment (128 bytes) there, and the warp reads
// them back so that 8 lanes hold one segment: each store instruction writes 4
// whole 128-byte lines.  (Each lane storing its own row touches 32 lines per
// instruction and took about twice as long; a shuffle transpose among lane
// groups of 4 touches 8 and spends more in shuffles than the staging costs.)
// bf16 rows go the same way, two 32-dim blocks (128 bytes) per thread at a
// time.  All global stores are 16 bytes wide: a 32-byte
// st.global.v8 in this routine was found to land only its first word in one
// build of the kernel.
__device__ __noinline__ void store_o_rows(const TcArgs& a, uint32_t o_addr, int rows_here, bool whole,
                                          int64_t out_base, int64_t piece_base, int r0, int d0, float inv,
                                          uint32_t stage) {
  const int lane = threadIdx.x & 31;
  const int h = lane >> 4, lr = lane & 15;          // this thread's half-row and row within the warp
  const int dbase = d0 - 128 * h;                   // this CTA's first dim
  const int c = lane & 7;                           // read-back: chunk c of segment 4 i + lane / 8
  if (whole && a.o_bf16) {
    // bf16 rows, staged like the fp32 ones: two 32-dim blocks (128 bytes) per
    // thread at a time
    __nv_bfloat16* const outb = static_cast<__nv_bfloat16*>(a.o_part) + out_base * kDv;
#pragma unroll 1
    for (int kp = 0; kp < 2; ++kp) {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {        // each 32-dim block: 4 of the row segment's 8 chunks
        uint32_t rr[32];
        tmem_ld16x2_sync<128>(o_addr + 32 * (2 * kp + half), rr);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          __nv_bfloat162 hh =
              __floats2bfloat162_rn(__uint_as_float(rr[2 * e]) * inv, __uint_as_float(rr[2 * e + 1]) * inv);
          w[e] = *reinterpret_cast<uint32_t*>(&hh);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_shared_v4(stage + (uint32_t)lr * kXRowBytes + ((uint32_t)((8 * h + 4 * half + i) ^ lr) << 4), w[4 * i],
                       w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int sg = 4 * i + (lane >> 3);         // segment: row sg / 2, half sg % 2
        const int sr = sg >> 1, sh = sg & 1;
        const uint4 v = ld_shared_v4(stage + (uint32_t)sr * kXRowBytes + ((uint32_t)((8 * sh + c) ^ sr) << 4));
        if (r0 + sr < rows_here)
          *reinterpret_cast<uint4*>(outb + (int64_t)(r0 + sr) * kDv + dbase + 128 * sh + 64 * kp + 8 * c) = v;
      }
      __syncwarp();
    }
    return;
  }
  float* const out0 = whole ? static_cast<float*>(a.o_part) + out_base * kDv : a.piece_o + piece_base * kDv;
#pragma unroll 1
  for (int k = 0; k < 4; ++k) {
    uint32_t rr[32];
    tmem_ld16x2_sync<128>(o_addr + 32 * k, rr);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      st_shared_v4(stage + (uint32_t)lr * kXRowBytes + ((uint32_t)((8 * h + i) ^ lr) << 4),
                   __float_as_uint(__uint_as_float(rr[4 * i]) * inv), __float_as_uint(__uint_as_float(rr[4 * i + 1]) * inv),
                   __float_as_uint(__uint_as_float(rr[4 * i + 2]) * inv), __float_as_uint(__uint_as_float(rr[4 * i + 3]) * inv));
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int sg = 4 * i + (lane >> 3);           // segment: row sg / 2, half sg % 2
      const int sr = sg >> 1, sh = sg & 1;
      const uint4 v = ld_shared_v4(stage + (uint32_t)sr * kXRowBytes + ((uint32_t)((8 * sh + c) ^ sr) << 4));
      if (r0 + sr < rows_here)
        *reinterpret_cast<uint4*>(out0 + (int64_t)(r0 + sr) * kDv + dbase + 128 * sh + 32 * k + 4 * c) = v;
    }
    __syncwarp();                                   // the reads are done before the next k's writes
  }
}

// ---------------------------------------------------------------------------- main kernel
// A 2-CTA cluster per (work range, row group).  CTA `rank` loads key/value dims
// [256 rank, 256 rank + 256) and 32 rope dims of every tile,
// computes its partial scores over them, swaps partial scores with its peer and
// accumulates its own 256 value dims of O.  Both CTAs walk the same tile
// sequence; the score exchange is double-buffered and S tiles are released as
// soon as they have been read, so QK products run up to two tiles ahead of the
// softmax while the exchange is in flight.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv,
                      const __grid_constant__ CUtensorMap tmap_q64, const __grid_constant__ CUtensorMap tmap_kv64,
                      const __grid_constant__ CUtensorMap tmap_kv4, TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // The layout needs a 1024-byte aligned base and the launch reserves no slack
  // for aligning it here: every CTA of the launch sees the same base, so a
  // misaligned one makes all of them stop at once, before any barrier.
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) flag(a.status, DCP_STATUS_INTERNAL);
    return;
  }
  // launched as a programmatic dependent of the plan kernel: nothing it wrote
  // (the tile prefix sums, the empty units' rows) is read before this
  griddep_wait();
  unsigned char* smem = smem_raw;
  const SmemLayout sl = smem_layout(a.Rg, a.nts);
  unsigned char* qc_s = smem + sl.qc;
  unsigned char* qr_s = smem + sl.qr;
  unsigned char* x_s = smem + sl.x;
  unsigned char* ring = smem + sl.ring;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bars);
  uint64_t* tfull = bars + kFixedBarSlots;      // tile slot landed
  uint64_t* tempty = tfull + kMaxTileSlots;     // tile slot released by its PV product
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
  const int nts = a.nts;
  int nhalf = 0;  // softmax warps with rows of the group (warp w < 8 serves rows 32 (w % 4) + 16 (w / 4) + [0, 16))
  for (int w = 0; w < 8; ++w) nhalf += 32 * (w & 3) + kHalfRows * (w >> 2) < Rg;
  const int32_t U = a.B * a.n_held;
  const int64_t T = a.tile_start[U];
  const int64_t lo = range_lo(T, v, a.V), hi = range_lo(T, v + 1, a.V);
  const uint32_t ntiles_cta = (uint32_t)(hi - lo);

  if (tid == 0) {
    *abort_s = 0;
    for (int i = 0; i < kNumFixedBars; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[kQFull], nhalf + 1);  // softmax warps + the query-chunk TMA
    mbar_init(&bars[kSFree0], nhalf);     // every softmax warp has read the partial scores
    mbar_init(&bars[kSFree1], nhalf);
    mbar_init(&bars[kPFull0], nhalf);
    mbar_init(&bars[kPFull1], nhalf);
    mbar_init(&bars[kOFree], nhalf);
    // The score exchange runs as one channel per softmax warp (its 16 rows), with
    // one single-arrival "landed" barrier per buffer and channel.
    for (int i = 0; i < nts; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 1);
    }
    fence_barrier_init();
    // tile j's partial scores from the peer land in buffer (j & 1) ^ 1: expect tiles 0 and 1
    for (uint32_t j = 0; j < 2 && j < ntiles_cta; ++j)
      for (int w = 0; w < 8; ++w)
        if (32 * (w & 3) + kHalfRows * (w >> 2) < Rg)
          mbar_arrive_expect_tx(&bars[kXFull + 8 * ((j & 1) ^ 1) + w], kHalfRows * kXRowBytes);
  }
  // rows of a page past a request's length are read with zero weight: start from finite zeros
  for (int i = tid; i < nts * kSlotBytes / 16; i += kThreads) reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  // query rows past the group are read by the M = 128 products: zeros
  for (int i = tid; i < (int)(sl.x / 16); i += kThreads) reinterpret_cast<uint4*>(qc_s)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before any remote store or arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    // The whole warp walks the tile sequence: its lanes fetch the block-table
    // entries of 32 tiles at a time (the next 32 are already in flight), lane 0
    // takes each tile's page ids by shuffle, waits for the ring slot and issues
    // the TMA copies.  Waits are lane-0 polls broadcast to the warp.
    if (lo < hi) {
      if (lane == 0) {
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_kv);
        prefetch_tmap(&tmap_q64);
        prefetch_tmap(&tmap_kv64);
        prefetch_tmap(&tmap_kv4);
      }
      SegIter it;
      it.init(a.tile_start, U, lo, hi);
      int32_t u, t0, nt, kslot;
      bool whole;
      uint32_t j = 0;  // tile index within this CTA's range
      int seg = 0;
      bool ok = true;
      const int nbox = kTile / a.box_rows;
      struct Boxes {
        int32_t y[8];
        uint32_t bytes;
      };
      auto box_y = [](const Boxes& bx, int q) -> int32_t {  // register-resident select (no local memory)
        int32_t y = bx.y[0];
#pragma unroll
        for (int i = 1; i < 8; ++i)
          if (q == i) y = bx.y[i];
        return y;
      };
      // lane l: page ids of the boxes of tile tile0 + l (-2: not needed, -1: past the table)
      auto fetch_batch = [&](int b, int64_t nvis, int32_t tile0, int32_t tile_end, int32_t (&pg)[8]) {
        // (local rows and pool rows fit in 32 bits: the host checks the pool size)
        const int32_t tile = tile0 + lane;
        const int32_t rho0 = tile * kTile;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          pg[q] = -2;
          const int32_t rho = rho0 + q * a.box_rows;
          if (tile < tile_end && q < nbox && rho < nvis) {
            const int32_t pidx = rho / a.L.P;
            pg[q] = pidx < a.max_pages ? __ldg(a.bt + (int64_t)b * a.bt_stride + pidx) : -1;
          }
        }
      };
      // lane l: pool rows of the boxes of tile tile0 + l from their page ids (-1: no box).
      // Which boxes are needed is recomputed here, not read from the -2 marks, so a
      // block-table entry of -2 is reported like any other bad page id.
      auto to_rows = [&](int rs, int32_t tile0, int32_t tile_end, int64_t nvis, const int32_t (&pg)[8],
                         int32_t (&yb)[8]) {
        const int32_t tile = tile0 + lane;
        const int32_t rho0 = tile * kTile;
        const int32_t pool0 = rs * (int32_t)a.pool_rows;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          yb[q] = -1;
          if (!(tile < tile_end && q < nbox && rho0 + q * a.box_rows < nvis)) continue;
          if (pg[q] < 0 || pg[q] >= a.pool_pages) {
            if (rank == 0) flag(a.status, DCP_STATUS_BAD_PAGE_ID);
            continue;
          }
          // a box never crosses a page: its height is min(P, 64) and it starts at a
          // multiple of it, so it starts a page when P <= 64
          const int32_t rho = rho0 + q * a.box_rows;
          const int32_t in_page = a.L.P <= kTile ? 0 : rho % a.L.P;
          yb[q] = pool0 + pg[q] * a.L.P + in_page;
        }
      };
      // the same rows without the bad-page report (the batch is checked again when it is issued)
      auto to_rows_quiet = [&](int rs, int32_t tile0, const int32_t (&pg)[8], int32_t (&yb)[8]) {
        const int32_t rho0 = (tile0 + lane) * kTile;
        const int32_t pool0 = rs * (int32_t)a.pool_rows;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int32_t rho = rho0 + q * a.box_rows;
          yb[q] = (pg[q] < 0 || pg[q] >= a.pool_pages) ? -1 : pool0 + pg[q] * a.L.P + (a.L.P <= kTile ? 0 : rho % a.L.P);
        }
      };
      auto make_boxes = [&](const int32_t (&y)[8], Boxes& bx) {
        bx.bytes = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          bx.y[q] = y[q];
          if (y[q] >= 0) bx.bytes += a.box_rows * 128;
        }
      };
      // one chunk (all its boxes) into `dst`; exactly as many TMA instructions as
      // boxes (predicated-off copies in an unrolled loop still cost issue time)
      auto issue_chunk = [&](const Boxes& bx, unsigned char* dst, uint64_t* bar, int k) {
        if (nbox == 1) {
          if (bx.y[0] >= 0) tma_load_2d(dst, &tmap_kv, bar, k * kChunkDims, bx.y[0]);
        } else {
          for (int q = 0; q < nbox; ++q) {
            const int32_t y = box_y(bx, q);
            if (y >= 0) tma_load_2d(dst + q * a.box_rows * 128, &tmap_kv, bar, k * kChunkDims, y);
          }
        }
      };
      // this CTA's 32 rope dims of the tile: rows of 64 bytes, 64-byte swizzle
      auto issue_rope = [&](const Boxes& bx, unsigned char* dst, uint64_t* bar) {
        const int32_t x = 2 * kOwnChunks * kChunkDims + kRopeHalf * (int)rank;
        if (nbox == 1) {
          if (bx.y[0] >= 0) tma_load_2d(dst, &tmap_kv64, bar, x, bx.y[0]);
        } else {
          for (int q = 0; q < nbox; ++q) {
            const int32_t y = box_y(bx, q);
            if (y >= 0) tma_load_2d(dst + q * a.box_rows * 64, &tmap_kv64, bar, x, y);
          }
        }
      };
      uint32_t ts = 0, tphase = 0;  // ring slot of tile j and its use parity
      auto load_tile = [&](const Boxes& bx) -> bool {
        if (!warp_wait(&tempty[ts], tphase ^ 1, abort_s, lane)) return false;
        if (lane == 0) {
          mbar_arrive_expect_tx(&tfull[ts], bx.bytes * kOwnChunks + bx.bytes / 2);
          unsigned char* dst = ring + ts * kSlotBytes;
          if (nbox == 1) {
            // all four value chunks of the tile with one 3-D box: [4 chunks][64 rows][128 B]
            if (bx.y[0] >= 0) tma_load_3d(dst, &tmap_kv4, &tfull[ts], 0, bx.y[0], kOwnChunks * (int)rank);
          } else {
            for (int i = 0; i < kOwnChunks; ++i)
              issue_chunk(bx, dst + i * kChunkBytes, &tfull[ts], kOwnChunks * (int)rank + i);
          }
          issue_rope(bx, dst + kRopeOff, &tfull[ts]);
        }
        ++j;
        if (++ts == (uint32_t)nts) {
          ts = 0;
          tphase ^= 1;
        }
        return true;
      };
      // A segment's length and the page ids of its first 32 tiles are loaded
      // during the segment before it, so that a segment start waits on no
      // global load.  The early page ids are read without the length (up to
      // max_pages entries of the row); to_rows applies the length when they are
      // used.
      bool have = it.next(&u, &t0, &nt, &whole, &kslot);
      int32_t pgf[8];       // page ids of the boxes of the segment's first 32 tiles
      int64_t nvis_f = 0;   // and its visible rows
      if (have) {
        bool bad0 = false;
        nvis_f = unit_nvis_max(a, u / a.n_held, u % a.n_held, &bad0);
        fetch_batch(u / a.n_held, INT64_MAX, t0, t0 + nt, pgf);
      }
      while (ok && have) {
        const int b = u / a.n_held, rs = u % a.n_held;
        const int64_t nvis = nvis_f;
        const int32_t t_end = t0 + nt;
        // block-table entries of the next 32 tiles are in flight while the
        // current 32 are issued; each lane turns its tile's entries into TMA rows
        int32_t pgn[8], yc[8], yn = -1;  // yn: next batch's first-box rows (L2 prefetch)
        to_rows(rs, t0, t_end, nvis, pgf, yc);
        fetch_batch(b, nvis, t0 + 32, t_end, pgn);
        // the next segment, peeked once this segment's first tile is issued (the
        // peek waits on the unit table): its length and first page ids are then
        // in flight during this segment
        SegIter nx = it;
        int32_t u2 = 0, t02 = 0, nt2 = 0, ks2 = 0;
        bool wh2 = false, has_next = false;
        int32_t y_next = -1;    // first-box row of the next segment's tile `lane` (L2 prefetch)
        bool next_rows = false;
        // the query's chunk 4r + 3 and its rope dims [32r, 32r + 32) for the SS part of QK
        if (!warp_wait(&bars[kQEmpty], (seg & 1) ^ 1, abort_s, lane)) { ok = false; break; }
        if (lane == 0) {
          const int32_t qy = b * a.R_total + g * Rg;
          mbar_arrive_expect_tx(&bars[kQFull], Rg * (2 * 128 + 64));
          for (int i = kQTmemChunks; i < kOwnChunks; ++i)
            tma_load_2d(qc_s + (i - kQTmemChunks) * 128 * 128, &tmap_q, &bars[kQFull],
                        (kOwnChunks * (int)rank + i) * kChunkDims, qy);
          tma_load_2d(qr_s, &tmap_q64, &bars[kQFull], 2 * kOwnChunks * kChunkDims + kRopeHalf * (int)rank, qy);
        }
        ++seg;
        for (int jj = 0; jj < nt && ok; ++jj) {
          if (jj > 0 && (jj & 31) == 0) {
            to_rows(rs, t0 + jj, t_end, nvis, pgn, yc);
            fetch_batch(b, nvis, t0 + jj + 32, t_end, pgn);
          }
          if (nbox == 1) {
            // The ring holds a few tiles, fewer than HBM latency times the tile
            // rate: each tile is also prefetched into L2 kL2Ahead tiles before its
            // ring load, so that the load finds it there.
            // The next batch's rows, once its block-table entries have arrived:
            if ((jj & 31) == 32 - kL2Ahead) {
              int32_t yt[8];
              to_rows_quiet(rs, t0 + jj + kL2Ahead, pgn, yt);
              yn = yt[0];
            }
            // tile jj + kL2Ahead into L2, so that its ring load finds it there
            const int32_t ja = jj + kL2Ahead;
            const int32_t ya = __shfl_sync(0xffffffffu, (ja & 31) > (jj & 31) ? yc[0] : yn, ja & 31);
            if (lane == 0 && ja < nt && ya >= 0) {
              tma_prefetch_3d(&tmap_kv4, 0, ya, kOwnChunks * (int)rank);
              tma_prefetch_2d(&tmap_kv64, 2 * kOwnChunks * kChunkDims + kRopeHalf * (int)rank, ya);
            }
            // past this segment's end: the next segment's first tiles
            if (ja >= nt && has_next && ja - nt < nt2 && ja - nt < 32) {
              if (!next_rows) {
                int32_t yt[8];
                to_rows_quiet(u2 % a.n_held, t02, pgf, yt);
                y_next = yt[0];
                next_rows = true;
              }
              const int32_t yb = __shfl_sync(0xffffffffu, y_next, ja - nt);
              if (lane == 0 && yb >= 0) {
                tma_prefetch_3d(&tmap_kv4, 0, yb, kOwnChunks * (int)rank);
                tma_prefetch_2d(&tmap_kv64, 2 * kOwnChunks * kChunkDims + kRopeHalf * (int)rank, yb);
              }
            }
          }
          Boxes cur;
          if (nbox == 1) {
            cur.y[0] = __shfl_sync(0xffffffffu, yc[0], jj & 31);
            cur.bytes = cur.y[0] >= 0 ? kTile * 128 : 0;
          } else {
            int32_t y[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) y[q] = __shfl_sync(0xffffffffu, yc[q], jj & 31);
            make_boxes(y, cur);
          }
          ok = load_tile(cur);
          if (jj == 0) {
            has_next = nx.next(&u2, &t02, &nt2, &wh2, &ks2);
            if (has_next) {
              bool bad2 = false;
              nvis_f = unit_nvis_max(a, u2 / a.n_held, u2 % a.n_held, &bad2);
              fetch_batch(u2 / a.n_held, INT64_MAX, t02, t02 + nt2, pgf);
            }
          }
        }
        it = nx;  // the segment just peeked (its fields below)
        have = has_next;
        u = u2, t0 = t02, nt = nt2, whole = wh2, kslot = ks2;
      }
      // Drain: every slot's last release (a tensor-core commit) lands before the
      // CTA may retire.  Bounded; skipped after an abort.
      if (ok) {
        for (uint32_t s = 0; s < (uint32_t)nts && s < ntiles_cta; ++s) {
          const uint32_t last = s + ((ntiles_cta - 1 - s) / nts) * nts;  // last tile in slot s
          if (!warp_wait(&tempty[s], (last / nts) & 1, abort_s, lane)) break;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ QK issuer
    if (lane == 0 && lo < hi) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, kTile, 0, 0);
      const uint64_t kdesc0 = sw128_desc(smem_u32(ring), 16, 1024);
      const uint64_t qcdesc0 = sw128_desc(smem_u32(qc_s), 16, 1024);
      const uint64_t qrdesc0 = sw64_desc(smem_u32(qr_s), 512);
      const uint64_t rdesc0 = sw64_desc(smem_u32(ring + kRopeOff), 512);
      // QK(j): query chunks 4r, 4r + 1 from TMEM (8 MMAs), chunks 4r + 2, 4r + 3
      // and the rope half from shared memory (8 + 2 MMAs), back to back.
      auto issue_qk = [&](uint32_t j, uint32_t ts) {
        const uint32_t d = tmem + kSCol + kTile * (j & 1);
        const uint32_t soff = (ts * kSlotBytes) >> 4;
        const uint64_t kd = kdesc0 + soff;
#pragma unroll
        for (int i = 0; i < kQTmemChunks; ++i)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(d, tmem + kQCol + 32 * i + 8 * kk, kd + i * (kChunkBytes >> 4) + 2 * kk, idesc_qk,
                        (i | kk) != 0);
#pragma unroll
        for (int i = kQTmemChunks; i < kOwnChunks; ++i)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(d, qcdesc0 + (i - kQTmemChunks) * ((128 * 128) >> 4) + 2 * kk,
                        kd + i * (kChunkBytes >> 4) + 2 * kk, idesc_qk, 1);
#pragma unroll
        for (int kk = 0; kk < kRopeHalf / 16; ++kk) mma_bf16_ss(d, qrdesc0 + 2 * kk, rdesc0 + soff + 2 * kk, idesc_qk, 1);
        mma_commit(&bars[kSFull0 + (j & 1)]);
      };
      // Two issuing threads, each blocking in order on its own conditions (no
      // polling loop): lane 0 of this warp issues QK(j) once tile j has landed
      // and the S tile it writes (last used by tile j - 2) has been read; lane 0
      // of warp kPvWarp issues PV(j) once P(j) is ready.  Both feed the same
      // in-order tensor pipe; each commit tracks its own thread's products.
      uint32_t ts_q = 0, ph_q = 0;  // ring slot of the next QK product and its use parity
      SegIter itq;
      itq.init(a.tile_start, U, lo, hi);
      int32_t uq, t0q, ntq, ksq;
      bool wq;
      uint32_t jq = 0;
      int q_seg = 0;
      bool ok = true;
      while (ok && itq.next(&uq, &t0q, &ntq, &wq, &ksq)) {
        for (int q_jj = 0; q_jj < ntq; ++q_jj, ++jq) {
          if (!mbar_wait(&bars[kSFree0 + (jq & 1)], ((jq >> 1) & 1) ^ 1, abort_s) ||
              (q_jj == 0 && !mbar_wait(&bars[kQFull], q_seg & 1, abort_s)) || !mbar_wait(&tfull[ts_q], ph_q, abort_s)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_qk(jq, ts_q);
          if (++ts_q == (uint32_t)nts) {
            ts_q = 0;
            ph_q ^= 1;
          }
          if (q_jj == ntq - 1) mma_commit(&bars[kQEmpty]);
        }
        ++q_seg;
      }
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0 && lo < hi) {
      const uint32_t idesc_pv = idesc_bf16_f32(128, 256, 0, 1);
      const uint64_t vdesc0 = sw128_desc(smem_u32(ring), kChunkBytes, 1024);
      SegIter itp;
      itp.init(a.tile_start, U, lo, hi);
      int32_t up, t0p, ntp, ksp;
      bool wp;
      uint32_t jp = 0, ts_p = 0;
      int p_seg = 0;
      bool ok = true;
      while (ok && itp.next(&up, &t0p, &ntp, &wp, &ksp)) {
        for (int p_jj = 0; p_jj < ntp; ++p_jj, ++jp) {
          // P(j) ready; the first product of a segment also needs the previous
          // segment's O read out
          if (!mbar_wait(&bars[kPFull0 + (jp & 1)], (jp >> 1) & 1, abort_s) ||
              (p_jj == 0 && p_seg >= 1 && !mbar_wait(&bars[kOFree], (p_seg - 1) & 1, abort_s))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pa = tmem + kPCol + 32 * (jp & 1);  // P(j): 64 bf16 = 32 columns
          const uint64_t vd = vdesc0 + ((ts_p * kSlotBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tmem + kOCol, pa + 8 * kk, vd + kk * (2048 >> 4), idesc_pv, !(p_jj == 0 && kk == 0));
          mma_commit(&tempty[ts_p]);
          mma_commit(&bars[kPVDone0 + (jp & 1)]);
          if (++ts_p == (uint32_t)nts) ts_p = 0;
        }
        ++p_seg;
      }
    }
  } else if (warp < 8 && 32 * (warp & 3) + kHalfRows * (warp >> 2) < Rg) {
    // ------------------------------------------------------------------ score exchange, softmax, epilogue
    // Warp w < 8 serves the 16 rows [r0, r0 + 16), r0 = 32 (w % 4) + 16 (w / 4),
    // with two threads per row: thread t takes row r0 + t % 16 and keys
    // [32 (t / 16), 32 (t / 16) + 32) of each tile (O columns [128 (t / 16), +128)).
    // Per tile j it reads its rows of this CTA's partial scores S_j^r, adds the
    // peer's (landed in buffer (j & 1) ^ 1) and runs the online softmax.  It also
    // ships its rows of S_j^r to the peer, from the registers it has just read
    // them into: staged in buffer j & 1 and sent with one bulk copy.  The buffer
    // is free: this warp read the peer's tile j - 1 out of it in the previous
    // tile, and my copy of tile j - 1 out of the peer's buffer had landed by
    // then.  Both conditions are local, so no barrier guards the buffers.
    // (Shipping S_{j+1} early, right after that read, was measured slower: the
    // extra TMEM read and staging sit in the middle of the softmax.)
    // Waits are warp-wide and bounded, so a timeout drains every thread.
    const int r0 = 32 * (warp & 3) + kHalfRows * (warp >> 2);
    const int ch = warp;  // exchange channel
    const int h = lane >> 4;
    const int row = r0 + (lane & 15);
    const uint32_t lane_addr = (uint32_t)r0 << 16;
    const uint32_t xrow = (uint32_t)row * kXRowBytes;
    if (lo < hi) {
      auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool { return warp_wait(bar, parity, abort_s, lane); };
      auto wwait_cluster = [&](uint64_t* bar, uint32_t parity) -> bool {
        return warp_wait_cluster(bar, parity, abort_s, lane);
      };
      const uint32_t peer = rank ^ 1u;
      const uint32_t x_peer = mapa_shared(smem_u32(x_s), peer);
      const uint32_t xfull_peer = mapa_shared(smem_u32(&bars[kXFull + ch]), peer);
      // this warp's rows of S_js (in registers) -> buffer js & 1 -> the peer's buffer (js & 1) ^ 1
      auto send = [&](uint32_t js, const uint32_t (&sv)[32]) {
        const uint32_t sb = js & 1;
        const uint32_t dst = smem_u32(x_s) + sb * sl.xbuf + xrow;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_shared_v4(dst + ((uint32_t)((8 * h + i) ^ (row & 15)) << 4), sv[4 * i], sv[4 * i + 1], sv[4 * i + 2],
                       sv[4 * i + 3]);
        fence_proxy_async_smem();  // the copy engine reads the staged rows
        __syncwarp();
        if (lane == 0)
          bulk_copy_to_peer(x_peer + (sb ^ 1) * sl.xbuf + (uint32_t)r0 * kXRowBytes,
                            x_s + sb * sl.xbuf + (uint32_t)r0 * kXRowBytes, kHalfRows * kXRowBytes,
                            xfull_peer + 8 * 8 * (sb ^ 1));
      };
      SegIter it;
      it.init(a.tile_start, U, lo, hi);
      int32_t u, t0, nt, kslot;
      bool whole;
      uint32_t jglob = 0;
      int seg = 0;
      bool ok = true;
      const int grow = g * Rg + row;
      const bool has_row = row < Rg && grow < a.R_total;
      // this warp's rows of the query chunks 4r, 4r + 1 (thread t: chunk t / 16 of
      // its row) for request b
      auto q_src = [&](int bq) {
        return reinterpret_cast<const uint4*>(a.q + ((int64_t)bq * a.R_total + grow) * kDk + 256 * (int)rank +
                                              kChunkDims * h);
      };
      // ... into TMEM for segment sq, once QK of segment sq - 1 no longer reads them
      auto load_q = [&](int bq, int sq) -> bool {
        if (!wwait(&bars[kQEmpty], (sq & 1) ^ 1)) return false;
        tc_fence_after();
        const uint4* src = q_src(bq);
        uint32_t r[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint4 w4 = has_row ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
          r[4 * k] = w4.x; r[4 * k + 1] = w4.y; r[4 * k + 2] = w4.z; r[4 * k + 3] = w4.w;
        }
        tmem_st16x2<32>(tmem + lane_addr + kQCol, r);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kQFull]);
        return true;
      };
      bool q_next = false;  // the next segment's query is already in TMEM
      // Each segment's description and length come from the segment before it
      // (peeked and loaded there), so a segment start waits on no global load.
      bool have = it.next(&u, &t0, &nt, &whole, &kslot);
      int64_t S_cur = have ? a.seq_lens[u / a.n_held] : 0;
      while (ok && have) {
        const int b = u / a.n_held, rs = u % a.n_held;
        if (!q_next && !load_q(b, seg)) { ok = false; break; }
        q_next = false;
        ++seg;
        // The next segment, peeked once this segment's first tile is done (the
        // peek waits on the unit table): its length is loaded then, its query
        // rows go into L2 then and into TMEM before this segment's epilogue, so
        // that its first QK product overlaps the epilogue.
        SegIter nx = it;
        int32_t u2 = 0, t02 = 0, nt2 = 0, ks2 = 0;
        bool wh2 = false, has_next = false;
        int64_t S_next = 0;
        const int64_t S = S_cur;
        int64_t nvis = 0;  // keys of this shard visible to the row
        if (has_row && S >= a.q_len) nvis = count_of(a.shard_begin + rs, S - a.q_len + grow / a.H + 1, a.L);
        float m_ref = -INFINITY;  // running maximum of the row (log2 units)
        float l = 0.f;            // this thread's half of the row's running sum
        float l_row = 0.f;        // the row's running sum
        for (int jj = 0; jj < nt; ++jj, ++jglob) {
          const uint32_t j = jglob, bsel = j & 1, rb = bsel ^ 1;
          // ---- this CTA's partial scores of tile j
          uint32_t s[32];  // score bits, keys [32 h, 32 h + 32)
          if (!wwait(&bars[kSFull0 + bsel], (j >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          tmem_ld16x2_sync<32>(tmem + lane_addr + kSCol + kTile * bsel, s);
          send(j, s);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kSFree0 + bsel]);
          // ---- the peer's partial scores of tile j: S = mine + peer's
          if (!wwait_cluster(&bars[kXFull + 8 * rb + ch], (j >> 1) & 1)) { ok = false; break; }
          {
            const uint32_t src = smem_u32(x_s) + rb * sl.xbuf + xrow;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 w4 = ld_shared_v4(src + ((uint32_t)((8 * h + i) ^ (row & 15)) << 4));
              const uint64_t a0 = f2_add(f2_pack(s[4 * i], s[4 * i + 1]), f2_pack(w4.x, w4.y));
              const uint64_t a1 = f2_add(f2_pack(s[4 * i + 2], s[4 * i + 3]), f2_pack(w4.z, w4.w));
              f2_unpack(a0, s[4 * i], s[4 * i + 1]);
              f2_unpack(a1, s[4 * i + 2], s[4 * i + 3]);
            }
          }
          __syncwarp();  // every lane's reads of buffer rb are done
          if (lane == 0 && j + 2 < ntiles_cta)
            mbar_arrive_expect_tx(&bars[kXFull + 8 * rb + ch], kHalfRows * kXRowBytes);
          // ---- online softmax of tile j
          const int64_t lim = nvis - ((int64_t)(t0 + jj) * kTile + 32 * h);  // keys k < lim are visible
          if (lim < 32) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (k >= lim) s[k] = __float_as_uint(-INFINITY);
          }
          float mx[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(s[k]);
#pragma unroll
          for (int k = 4; k < 32; k += 2)
            mx[((k - 4) >> 1) & 3] = fmax3(mx[((k - 4) >> 1) & 3], __uint_as_float(s[k]), __uint_as_float(s[k + 1]));
          float mraw = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
          mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 16));  // the row's other 32 keys
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
          if (__any_sync(0xffffffffu, need)) {
            // rows whose maximum moved: scale their O row once PV(j - 1) is done
            // (a row's maximum is finite only after a tile of this segment, so j >= 1)
            if (!wwait(&bars[kPVDone0 + ((j - 1) & 1)], ((j - 1) >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            rescale_rows(tmem + lane_addr + kOCol, alpha);
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          const float cs = a.scale_log2;
          const uint64_t cs2 = f2_pack(__float_as_uint(cs), __float_as_uint(cs));
          const uint64_t nm2 = f2_pack(__float_as_uint(-m_use), __float_as_uint(-m_use));
          uint64_t ps[4] = {0, 0, 0, 0};  // pairs of partial row sums (+0.f bits)
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            uint32_t x0, x1;
            f2_unpack(f2_fma(f2_pack(s[2 * k], s[2 * k + 1]), cs2, nm2), x0, x1);
            const float p0 = fast_exp2(__uint_as_float(x0));
            const float p1 = fast_exp2(__uint_as_float(x1));
            ps[k & 3] = f2_add(ps[k & 3], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
            __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
            pk[k] = *reinterpret_cast<uint32_t*>(&hh);
          }
          {
            uint32_t a0, a1;
            f2_unpack(f2_add(f2_add(ps[0], ps[1]), f2_add(ps[2], ps[3])), a0, a1);
            l = l * alpha + (__uint_as_float(a0) + __uint_as_float(a1));
          }
          // P(j) -> TMEM (A operand of the PV product) once PV(j - 2) has read the buffer
          if (j >= 2 && !wwait(&bars[kPVDone0 + bsel], ((j - 2) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          tmem_st16x2_16<16>(tmem + lane_addr + kPCol + 32 * bsel, pk);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kPFull0 + bsel]);
          if (jj == 0) {
            has_next = nx.next(&u2, &t02, &nt2, &wh2, &ks2);
            if (has_next) {
              S_next = a.seq_lens[u2 / a.n_held];
              if (has_row) asm volatile("prefetch.global.L2 [%0];" ::"l"(q_src(u2 / a.n_held)));
            }
          }
        }
        if (!ok) break;
        if (has_next) {
          if (!load_q(u2 / a.n_held, seg)) { ok = false; break; }
          q_next = true;
        }
        l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);
        // ---------------- epilogue: O rows / l -> o (this CTA's 256 dims), lse
        const uint32_t jl = jglob - 1;
        if (!wwait(&bars[kPVDone0 + (jl & 1)], (jl >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const int rows_here = min(Rg, a.R_total - g * Rg);
        const bool writes = row < rows_here;
        const int64_t out_base = ((int64_t)rs * a.B + b) * a.R_total + g * Rg;
        const int64_t piece_base = (int64_t)(2 * v + kslot) * a.R_total + g * Rg;
        const int64_t out_row = out_base + row, piece_row = piece_base + row;
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        // staging for the fp32 rows: this warp's rows of the buffer the last tile's
        // peer scores were read from
        store_o_rows(a, tmem + lane_addr + kOCol, rows_here, whole, out_base, piece_base, r0, 256 * (int)rank + 128 * h,
                     inv, smem_u32(x_s) + ((jl & 1) ^ 1) * sl.xbuf + (uint32_t)r0 * kXRowBytes);
        if (writes && h == 0 && rank == 0) {
          const float lse2 = l_row > 0.f ? m_ref + log2f(l_row) : -INFINITY;
          if (whole)
            a.lse_part[out_row] = a.base2 ? lse2 : lse2 * kLn2;
          else
            a.piece_lse[piece_row] = lse2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kOFree]);
        it = nx;  // the segment just peeked (its fields below)
        have = has_next;
        u = u2, t0 = t02, nt = nt2, whole = wh2, kslot = ks2;
        S_cur = S_next;
      }
    }
  }
  else if (warp < 8) {
    // No rows of the group: zero this warp's 16 TMEM lanes of the P and query
    // columns once, so the M = 128 products carry zeros, not stale data, in the
    // padding rows (their results are never read).
    const uint32_t zl = (uint32_t)(32 * (warp & 3) + kHalfRows * (warp >> 2)) << 16;
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    tmem_st16x2<32>(tmem + zl + kPCol, z);
    tmem_st16x2<32>(tmem + zl + kQCol, z);
    tmem_st_wait();
  }

  if (*abort_s && tid == 0) flag(a.status, DCP_STATUS_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  // The peer may still have stores or arrivals addressed to this CTA's shared
  // memory; retire the pair together.  After an abort, allow in-flight tensor
  // core commits (microseconds) to land first.
  if (*abort_s) __nanosleep(100000);
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------- fixup
// Merges the pieces of units cut by range boundaries (the same LSE rule as the
// shard merge, base 2).  Only range boundaries cut units, so block column k
// serves boundary k (between ranges k and k + 1): the unit containing that
// boundary's first tile, if the boundary falls inside it and no earlier boundary
// does (the first boundary inside a unit merges all its pieces).  Blocks per
// column: up to 12, each taking chunks of 8 query rows; thread 0 builds the
// unit's piece list in shared memory, then one warp per row merges the pieces
// with 16-byte loads and stores (lane l owns dims [16 l, 16 l + 16)).
constexpr int kFixupThreads = 256;
constexpr int kMaxPieces = 512;

constexpr int kFixupRows = kFixupThreads / 32;  // query rows per block: one per warp

__global__ void __launch_bounds__(kFixupThreads) fixup_kernel(TcArgs a) {
  __shared__ int32_t piece_s[kMaxPieces];
  __shared__ int32_t npiece_s, unit_s;
  griddep_wait();  // a programmatic dependent of the partial kernel: its pieces are complete after this
  const int32_t U = a.B * a.n_held;
  const int V = a.V;
  const int64_t T = a.tile_start[U];
  const int row0 = blockIdx.y * kFixupRows + (threadIdx.x >> 5);  // this warp's first query row
  const int row_step = gridDim.y * kFixupRows;
  const int lane = threadIdx.x & 31;
  auto store_row = [&](int64_t orow, const float (&v)[16]) {
    if (a.o_bf16) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o_part) + orow * kDv + 16 * lane);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __nv_bfloat162 t = __floats2bfloat162_rn(v[8 * h + 2 * i], v[8 * h + 2 * i + 1]);
          w[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        dst[h] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.o_part) + orow * kDv + 16 * lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  };
  if (threadIdx.x == 0) {
    const int k = blockIdx.x;
    const int64_t x = range_lo(T, k + 1, V);  // the boundary's first tile
    int unit = -1;
    if (x > 0 && x < T) {
      int32_t l = 0, h = U;  // the unit u with start[u] <= x < start[u + 1]
      while (h - l > 1) {
        const int32_t m = (l + h) >> 1;
        if (a.tile_start[m] <= x) l = m; else h = m;
      }
      const int64_t su = a.tile_start[l];
      if (su < x && (k == 0 || range_lo(T, k, V) <= su)) unit = l;
    }
    unit_s = unit;
  }
  __syncthreads();
  const int32_t u = unit_s;
  if (u < 0) return;
  const int b = u / a.n_held, rs = u % a.n_held;
  const int64_t s = a.tile_start[u], e = a.tile_start[u + 1];
  const int64_t out_row0 = ((int64_t)rs * a.B + b) * a.R_total;
  if (threadIdx.x == 0) {
    auto part_of = [&](int64_t x) {  // range containing tile x
      int vv = (int)((x * V) / T);
      while (vv + 1 < V && range_lo(T, vv + 1, V) <= x) ++vv;
      while (vv > 0 && range_lo(T, vv, V) > x) --vv;
      return vv;
    };
    const int v0 = part_of(s), v1 = part_of(e - 1);
    int n = 0;
    if (v0 != v1) {
      for (int vv = v0; vv <= v1 && n < kMaxPieces; ++vv) {
        const int64_t rlo = range_lo(T, vv, V);
        if (rlo == range_lo(T, vv + 1, V)) continue;  // empty range: no piece
        piece_s[n++] = 2 * vv + (rlo >= s ? 0 : 1);
      }
    }
    npiece_s = n;
  }
  __syncthreads();
  const int np = npiece_s;
  for (int row = row0; row < a.R_total; row += row_step) {
    // Pieces two at a time: both pieces' lse and o loads are issued before
    // either is used (the row's loads are one latency, not one per piece).
    float m = -INFINITY;
    for (int k = 0; k < np; ++k) m = fmaxf(m, a.piece_lse[(int64_t)piece_s[k] * a.R_total + row]);
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int k = 0; k < np; k += 2) {
        const bool two = k + 1 < np;
        const int64_t pr0 = (int64_t)piece_s[k] * a.R_total + row;
        const int64_t pr1 = two ? (int64_t)piece_s[k + 1] * a.R_total + row : pr0;
        const float4* src0 = reinterpret_cast<const float4*>(a.piece_o + pr0 * kDv + 16 * lane);
        const float4* src1 = reinterpret_cast<const float4*>(a.piece_o + pr1 * kDv + 16 * lane);
        float4 o0[4], o1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o0[i] = src0[i];
          o1[i] = src1[i];
        }
        const float l0 = a.piece_lse[pr0];
        const float l1 = two ? a.piece_lse[pr1] : -INFINITY;
        const float w0 = l0 == -INFINITY ? 0.f : exp2f(l0 - m);
        const float w1 = l1 == -INFINITY ? 0.f : exp2f(l1 - m);
        wsum += w0 + w1;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[4 * i] = fmaf(w1, o1[i].x, fmaf(w0, o0[i].x, acc[4 * i]));
          acc[4 * i + 1] = fmaf(w1, o1[i].y, fmaf(w0, o0[i].y, acc[4 * i + 1]));
          acc[4 * i + 2] = fmaf(w1, o1[i].z, fmaf(w0, o0[i].z, acc[4 * i + 2]));
          acc[4 * i + 3] = fmaf(w1, o1[i].w, fmaf(w0, o0[i].w, acc[4 * i + 3]));
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= inv;
    store_row(out_row0 + row, acc);
    if (lane == 0) {
      const float lse2 = wsum > 0.f ? m + log2f(wsum) : -INFINITY;
      a.lse_part[out_row0 + row] = a.base2 ? lse2 : lse2 * kLn2;
    }
  }
}

// ---------------------------------------------------------------------------- host side
struct Plan {
  int Rg, ngroups, V, nts, box_rows;
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

SmemLimit g_partial_smem;  // partial_tc_kernel's dynamic shared-memory limit, per device

// Resident 2-CTA clusters of partial_tc_kernel at `smem` bytes on the current
// device.  Cached per device and shared-memory size (a workload uses one or two
// sizes); guarded by a mutex, since one host thread per GPU may plan at once.
int max_active_clusters(size_t smem) {
  constexpr int kEntries = 8;
  struct Entry {
    size_t smem;
    int clusters;
  };
  static std::mutex m;
  static Entry cache[kMaxDevices][kEntries] = {};
  const int dev = current_device();
  if (dev < 0) return 0;
  {
    std::lock_guard<std::mutex> lock(m);
    for (const Entry& e : cache[dev])
      if (e.smem == smem && e.clusters > 0) return e.clusters;
  }
  if (!g_partial_smem.ensure(reinterpret_cast<const void*>(&partial_tc_kernel), smem)) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 512, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, partial_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (n > 0) {
    std::lock_guard<std::mutex> lock(m);
    Entry* slot = &cache[dev][0];
    for (Entry& e : cache[dev])
      if (e.clusters == 0 || e.smem == smem) {
        slot = &e;
        break;
      }
    *slot = Entry{smem, n};
  }
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
  const size_t budget = 232448;  // 227 KB
  int nts = (int)((budget - base.total) / kSlotBytes);
  if (nts > kMaxTileSlots) nts = kMaxTileSlots;
  p->nts = nts;
  p->smem = smem_layout(p->Rg, nts).total;
  // clusters that can be resident at once (both CTAs of a cluster share a GPC)
  const int clusters = max_active_clusters(p->smem);
  if (clusters > 0) {
    // V ranges per row group.  One wave of V0 = clusters / ngroups ranges is the
    // default; when that leaves many clusters idle (ngroups not much below the
    // cluster count, e.g. a chunked extend's many row groups), a larger V run
    // in several waves finishes sooner: the time is waves / V of one group's
    // whole sequence.  A larger V must gain 5 % to pay for its cut units.
    const int V0 = clusters / p->ngroups > 1 ? clusters / p->ngroups : 1;
    auto cost = [&](int Vc) {
      return (double)(((int64_t)Vc * p->ngroups + clusters - 1) / clusters) / Vc;
    };
    int best = V0;
    for (int Vc = V0 + 1; Vc <= 8; ++Vc)
      if (cost(Vc) < 0.95 * cost(best)) best = Vc;
    p->V = best;
  }
  const int P = layout->page_size;
  p->box_rows = P >= kTile ? kTile : P;
  const int64_t U = (int64_t)B * n_held;
  p->ws_start_bytes = align256((size_t)(U + 1) * 4);
  // With one range per row group no unit is cut, so no piece is ever written.
  p->ws_piece_o_bytes = p->V > 1 ? align256((size_t)2 * p->V * R_total * kDv * 4) : 0;
  p->ws_piece_lse_bytes = p->V > 1 ? align256((size_t)2 * p->V * R_total * 4) : 0;
  p->ws_total = p->ws_start_bytes + p->ws_piece_o_bytes + p->ws_piece_lse_bytes;
  return nts >= 3;
}

// bf16 [rows, 576] row-major, boxes of [box_rows, 64] with 128-byte swizzle, or
// (half = true) boxes of [box_rows, 32] with 64-byte swizzle
// bf16 [rows, 576] seen as [9 chunks][rows][64 dims] (dims innermost, then rows,
// then chunks 128 bytes apart): boxes of [4 chunks][box_rows][64] land as four
// consecutive 128-byte-swizzled [box_rows][64] tiles.
bool make_tmap_chunks(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kChunkDims, (cuuint64_t)rows, (cuuint64_t)(kDk / kChunkDims)};
  cuuint64_t strides[2] = {(cuuint64_t)kDk * 2, (cuuint64_t)kChunkDims * 2};
  cuuint32_t box[3] = {(cuuint32_t)kChunkDims, box_rows, (cuuint32_t)kOwnChunks};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows, bool half = false) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDk, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDk * 2};
  cuuint32_t box[2] = {(cuuint32_t)(half ? kRopeHalf : kChunkDims), box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, half ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool page_size_ok(int P) { return P >= 8 && P % 8 == 0 && (P % kTile == 0 || kTile % P == 0); }

}  // namespace

extern "C" size_t dcp_mla_decode_workspace_size(const dcp_layout_t* layout, int32_t shard_begin,
                                                int32_t shard_end, int32_t B, int32_t q_len, int32_t H) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end ||
      B < 1 || q_len < 1 || H < 1 || (int64_t)q_len * H > kMaxQueryRows)
    return 0;
  Plan p;
  if (!make_plan(layout, shard_end - shard_begin, B, q_len, H, &p)) return 0;
  return p.ws_total;
}

namespace {

// Host checks of dcp_mla_decode_partial's arguments (all but the workspace).
int32_t check_decode_args(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end, const void* q,
                          int32_t B, int32_t q_len, int32_t H, const void* arena, int64_t pool_pages,
                          const int32_t* block_table, int64_t bt_stride, int64_t max_pages, const int64_t* seq_lens,
                          float scale, int32_t lse_base, const void* o_part, int32_t o_part_dtype,
                          const float* lse_part) {
  if (!layout_ok(layout) || shard_begin < 0 || shard_end > layout->n_shards || shard_begin >= shard_end)
    return DCP_ERR_INVALID;
  if (B < 1 || q_len < 1 || H < 1 || (int64_t)q_len * H > kMaxQueryRows) return DCP_ERR_INVALID;
  if (pool_pages < 1 || max_pages < 1 || bt_stride < max_pages) return DCP_ERR_INVALID;
  if (!q || !arena || !block_table || !seq_lens || !o_part || !lse_part) return DCP_ERR_INVALID;
  if (o_part_dtype != DCP_F32 && o_part_dtype != DCP_BF16) return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (!(scale > 0.f) || !(scale < INFINITY)) return DCP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(arena) |
       reinterpret_cast<uintptr_t>(o_part)) & 15)
    return DCP_ERR_INVALID;
  if (!page_size_ok(layout->page_size)) return DCP_ERR_UNSUPPORTED;
  const int64_t pool_rows = pool_pages * layout->page_size;
  const int64_t n_held = shard_end - shard_begin;
  if (n_held * pool_rows >= INT32_MAX || (int64_t)B * q_len * H >= INT32_MAX || (int64_t)B * n_held >= INT32_MAX / 2)
    return DCP_ERR_UNSUPPORTED;
  return DCP_OK;
}

// Tensor maps and the three launches of one partial decode on a checked plan and
// a workspace of at least p.ws_total bytes (256-byte aligned).
int32_t launch_decode(const Plan& p, const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                      const void* q, int32_t B, int32_t q_len, int32_t H, const void* arena, int64_t pool_pages,
                      const int32_t* block_table, int64_t bt_stride, int64_t max_pages, const int64_t* seq_lens,
                      float scale, int32_t lse_base, void* o_part, int32_t o_part_dtype, float* lse_part,
                      void* workspace, int32_t* status, void* stream) {
  const int n_held = shard_end - shard_begin;
  const int64_t pool_rows = pool_pages * layout->page_size;
  CUtensorMap tq, tkv, tq64, tkv64, tkv4;
  if (!make_tmap(&tq, q, (uint64_t)B * q_len * H, (uint32_t)p.Rg)) return DCP_ERR_CUDA;
  if (!make_tmap(&tkv, arena, (uint64_t)n_held * pool_rows, (uint32_t)p.box_rows)) return DCP_ERR_CUDA;
  if (!make_tmap(&tq64, q, (uint64_t)B * q_len * H, (uint32_t)p.Rg, true)) return DCP_ERR_CUDA;
  if (!make_tmap(&tkv64, arena, (uint64_t)n_held * pool_rows, (uint32_t)p.box_rows, true)) return DCP_ERR_CUDA;
  if (!make_tmap_chunks(&tkv4, arena, (uint64_t)n_held * pool_rows, (uint32_t)p.box_rows)) return DCP_ERR_CUDA;
  if (!g_partial_smem.ensure(reinterpret_cast<const void*>(&partial_tc_kernel), p.smem)) return DCP_ERR_CUDA;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  TcArgs a;
  a.L = to_layout(layout);
  a.shard_begin = shard_begin;
  a.n_held = n_held;
  a.B = B; a.q_len = q_len; a.H = H; a.R_total = q_len * H;
  a.Rg = p.Rg; a.ngroups = p.ngroups; a.V = p.V; a.nts = p.nts; a.box_rows = p.box_rows;
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
  // The partial kernel and the fixup are programmatic dependent launches: each
  // grid may be scheduled while the one before it finishes, and waits
  // (griddepcontrol.wait) before it reads anything that one wrote.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(2 * p.V * p.ngroups));
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = p.smem;
  lc.stream = st;
  lc.attrs = pdl;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, partial_tc_kernel, tq, tkv, tq64, tkv64, tkv4, a) != cudaSuccess) return DCP_ERR_CUDA;
  // Cut units need their pieces merged: one block column per range boundary,
  // one warp per row up to 96 rows, blocks looping over further row chunks.
  // With one range per row group nothing is cut and no fixup runs.
  if (p.V > 1) {
    const unsigned fix_y = (unsigned)std::min((a.R_total + kFixupRows - 1) / kFixupRows, 12);
    cudaLaunchConfig_t lf = {};
    lf.gridDim = dim3((unsigned)(p.V - 1), fix_y);
    lf.blockDim = dim3(kFixupThreads);
    lf.stream = st;
    lf.attrs = pdl;
    lf.numAttrs = 1;
    if (cudaLaunchKernelEx(&lf, fixup_kernel, a) != cudaSuccess) return DCP_ERR_CUDA;
    return launch_status(3);
  }
  return launch_status(2);
}

}  // namespace

extern "C" int32_t dcp_mla_decode_partial(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                                          const void* q, int32_t B, int32_t q_len, int32_t H,
                                          const void* arena, int64_t pool_pages,
                                          const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                                          const int64_t* seq_lens, float scale, int32_t lse_base,
                                          void* o_part, int32_t o_part_dtype, float* lse_part,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* status, void* stream) {
  const int32_t rc = check_decode_args(layout, shard_begin, shard_end, q, B, q_len, H, arena, pool_pages,
                                       block_table, bt_stride, max_pages, seq_lens, scale, lse_base, o_part,
                                       o_part_dtype, lse_part);
  if (rc != DCP_OK) return rc;
  Plan p;
  if (!make_plan(layout, shard_end - shard_begin, B, q_len, H, &p)) return DCP_ERR_CUDA;
  if (!workspace || workspace_bytes < p.ws_total) return DCP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return DCP_ERR_INVALID;
  return launch_decode(p, layout, shard_begin, shard_end, q, B, q_len, H, arena, pool_pages, block_table, bt_stride,
                       max_pages, seq_lens, scale, lse_base, o_part, o_part_dtype, lse_part, workspace, status,
                       stream);
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

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_partial_scratch on the current device (looked up once per
// device; in host code the array's name is only a host-side stand-in).
void* scratch_address() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
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
  const int32_t rc = check_decode_args(layout, shard_begin, shard_end, q, B, q_len, H, arena, pool_pages,
                                       block_table, bt_stride, max_pages, seq_lens, scale, lse_base, o_part,
                                       o_part_dtype, lse_part);
  if (rc != DCP_OK) return rc;
  Plan p;
  if (!make_plan(layout, shard_end - shard_begin, B, q_len, H, &p)) return DCP_ERR_CUDA;
  if (p.ws_total > kStaticScratchBytes) return DCP_ERR_TOO_LARGE;
  void* ws = scratch_address();
  if (!ws) return DCP_ERR_CUDA;
  return launch_decode(p, layout, shard_begin, shard_end, q, B, q_len, H, arena, pool_pages, block_table, bt_stride,
                       max_pages, seq_lens, scale, lse_base, o_part, o_part_dtype, lse_part, ws, status, stream);
}
