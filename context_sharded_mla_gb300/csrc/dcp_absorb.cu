// dcp_absorb.cu — the two absorption products on either side of the decode
// path, on the sm_103a tensor cores.
//
// Sources: "MLA 的 Decode Context Parallelism", section 2 (identity 1: the K
// up-projection moves into the query, q_hat_h = q^C W^UK_h in R^512; identity
// 2: the V up-projection is applied once to the attention output);
// "Decode Context Parallelism" (zdszero), section "decode 路径：以 Kimi K3 的
// MLA 为例" (w_kc [H, 128, 512] and w_vc [H, 512, 128] split out of
// kv_b_proj; bmm(q_nope, w_kc) -> [B, H, 512] before attention,
// bmm(O, w_vc) -> [B, H, 128] after the merge).
//
// One kernel template computes, for head h, a tile of up to 128 query tokens
// starting at t0 and output columns [n0, n0 + NT):
//     D[t, n] = sum_k A[t, h, k] * W[h, k, n]
//   query side   A = q_nope (K = 128), W = w_kc (N = 512), NT = 256, two CTAs
//                per head; the epilogue writes bf16 into dims [0, 512) of the
//                576-d query rows, and the n0 = 0 CTA copies q_pe into dims
//                [512, 576)
//   output side  A = o (K = 512, bf16 or f32), W = w_vc (N = 128), NT = 128
// Per CTA, 192 threads:
//   warps 0-3  epilogue: warp w owns TMEM lanes (tokens) 32w .. 32w + 31.  For
//              an f32 A they first convert every K-step of A to bf16 and write
//              it into shared memory in the tensor core's 128-byte-swizzled
//              K-major layout (kind::f16 takes A and B of one type).
//   warp 4     TMA producer: per K-step of 64, A [128 tokens][64] as one 3-D
//              box over (k, head, token) (tokens past T read as zeros) and W
//              [64 k][NT] as NT/64 boxes of [64 k][64 n] (MN-major operand).
//   warp 5     TMEM owner and MMA issuer (one thread): four M=128, N=NT, K=16
//              products per K-step into NT fp32 TMEM columns.
// The decode batch T is small next to the weights (64 tokens x 96 heads
// against 12.6 MB of w_kc), so each product is bound by the HBM reads of the
// weights and activations, not by the tensor core (2T flops per weight element,
// 128 flops per byte at T = 64, under the bf16 ridge of about 280).
#include <cudaTypedefs.h>

#include <mutex>

#include "dcp_internal.cuh"
#include "sm100_ptx.cuh"

using namespace dcp;
using namespace dcp::sm100;

namespace {

constexpr int kAbsThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kIssuerWarp = 5;
constexpr int kKStep = 64;                    // K elements per pipeline stage
constexpr int kTokTile = 128;                 // tokens per CTA (MMA M)
constexpr uint32_t kATileBytes = kTokTile * kKStep * 2;   // 16 KB
constexpr uint32_t kWBoxBytes = kKStep * 64 * 2;          // one [64 k][64 n] box, 8 KB
// Output columns per CTA.  Narrower tiles (128 / 64 columns: 4 / 2 CTAs per
// head, 3 / 2 CTAs per SM) measured 12 % / 9 % slower at the K3 shapes: more
// CTAs start later and re-read the activations.
constexpr int kQTile = 256;                   // query side: 2 CTAs per head, 96 KB shared each
constexpr int kOTile = 128;                   // output side: 1 CTA per head
constexpr int kOStages = 6;                   // output side: 6 of its 8 K-steps in flight, 192 KB shared

template <int NT, int KSTEPS, int STAGES>
struct AbsorbSmem {
  static constexpr uint32_t kStage = kATileBytes + NT / 64 * kWBoxBytes;
  static constexpr uint32_t kBars = STAGES * kStage;        // full[STAGES], empty[STAGES], done
  static constexpr uint32_t kMisc = kBars + (2 * STAGES + 1) * 8;
  static constexpr uint32_t kBytes = kMisc + 16 + 1024;    // + alignment slack
};

struct AbsorbArgs {
  int64_t T;              // query tokens (B x q_len)
  int32_t H;
  const float* a_f32;     // f32 A [T, H, K] (output side only), else null
  int64_t a_f32_stride;   // elements between (t, h) rows of a_f32
  void* out;              // query side: bf16 [T, H, 576]; output side: [T, H, 128]
  int32_t out_bf16;       // output side: 1 -> bf16, 0 -> f32
  const __nv_bfloat16* q_pe;   // query side: bf16 rope part, 64 used per (t, h) row
  int64_t q_pe_stride;
  int32_t* status;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v2(uint32_t saddr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(saddr), "r"(a), "r"(b) : "memory");
}

// Bounded wait by a whole warp; every lane returns the same answer.
__device__ __forceinline__ bool warp_wait_all(uint64_t* bar, uint32_t parity, volatile int* abort_s) {
  const bool ok = mbar_wait(bar, parity, abort_s);
  return __all_sync(0xffffffffu, ok);
}

// kQuery: query side (bf16 A by TMA, bf16 output into 576-d rows + q_pe copy).
// kAF32: output side with an f32 A converted in the kernel.
template <int NT, int KSTEPS, int STAGES, bool kQuery, bool kAF32>
__global__ void __launch_bounds__(kAbsThreads, 1)
    absorb_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                  AbsorbArgs a) {
  using L = AbsorbSmem<NT, KSTEPS, STAGES>;
  constexpr int kNBoxes = NT / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* empty = full + STAGES;
  uint64_t* done = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * NT;
  const int h = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.z * kTokTile;

  // One K-step of loads into stage ks % STAGES (producer thread only).
  auto issue_loads = [&](int ks) {
    const int s = ks % STAGES;
    uint8_t* st = smem + s * L::kStage;
    mbar_arrive_expect_tx(&full[s], (kAF32 ? 0u : kATileBytes) + kNBoxes * kWBoxBytes);
    if (!kAF32) tma_load_3d(st, &tmap_a, &full[s], ks * kKStep, h, (int32_t)t0);
#pragma unroll
    for (int j = 0; j < kNBoxes; ++j)
      tma_load_3d(st + kATileBytes + j * kWBoxBytes, &tmap_w, &full[s], n0 + 64 * j, ks * kKStep, h);
  };

  // The producer initialises the barriers and puts the first STAGES K-steps in
  // flight at once, so their memory latency overlaps the TMEM allocation and
  // the CTA barrier below.
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_w);
    if (!kAF32) prefetch_tmap(&tmap_a);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kAF32 ? 1 + 4 : 1);   // producer (+ one arrival per converting warp)
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_s = 0;
    fence_barrier_init();
    for (int ks = 0; ks < STAGES && ks < KSTEPS; ++ks) issue_loads(ks);
  }
  if (warp == kIssuerWarp) {
    tmem_alloc(tmem_slot, NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int ks = STAGES; ks < KSTEPS; ++ks) {
        if (!mbar_wait(&empty[ks % STAGES], ((ks / STAGES) - 1) & 1, abort_s)) break;
        issue_loads(ks);
      }
    }
  } else if (warp == kIssuerWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTokTile, NT, 0, 1);
      bool ok = true;
      for (int ks = 0; ks < KSTEPS && ok; ++ks) {
        const int s = ks % STAGES;
        if (!mbar_wait(&full[s], (ks / STAGES) & 1, abort_s)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * L::kStage);
        const uint64_t adesc = sw128_desc(sa, 16, 1024);
        const uint64_t wdesc = sw128_desc(sa + kATileBytes, kWBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kKStep / 16; ++kk)
          mma_bf16_ss(tmem, adesc + kk * (32 >> 4), wdesc + kk * (2048 >> 4), idesc, (ks | kk) != 0);
        mma_commit(&empty[s]);
      }
      if (ok) mma_commit(done);
    }
  } else {
    // ------------------------------------------------------------------ warps 0-3
    const int row = tid;                        // this thread's token within the tile
    const int64_t t = t0 + row;
    bool ok = true;
    if (kQuery && n0 == 0 && t < a.T) {
      // the rope dims pass through: copy them while the product runs
      const uint4* src = reinterpret_cast<const uint4*>(a.q_pe + (t * a.H + h) * a.q_pe_stride);
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + (t * a.H + h) * kDk + kDv);
      uint4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __ldg(src + i);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = x[i];
    }
    if (kAF32) {
      // Convert A to bf16 into the swizzled K-major stage layout: 16-byte chunk c
      // of row r sits at r * 128 + ((c ^ (r % 8)) * 16) (tile base 1024-aligned).
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int s = ks % STAGES;
        if (ks >= STAGES && !warp_wait_all(&empty[s], ((ks / STAGES) - 1) & 1, abort_s)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + s * L::kStage);
        float4 v[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const int j = tid + 128 * m, r = j >> 4, c4 = j & 15;
          const int64_t tr = t0 + r;
          v[m] = tr < a.T ? __ldg(reinterpret_cast<const float4*>(a.a_f32 + (tr * a.H + h) * a.a_f32_stride +
                                                                   ks * kKStep + 4 * c4))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const int j = tid + 128 * m, r = j >> 4, c4 = j & 15;
          const uint32_t off = r * 128 + (((c4 >> 1) ^ (r & 7)) << 4) + (c4 & 1) * 8;
          st_shared_v2(sa + off, pack_bf16x2(v[m].x, v[m].y), pack_bf16x2(v[m].z, v[m].w));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
    // Epilogue: wait for the last product, then TMEM -> registers -> global.
    if (ok) ok = warp_wait_all(done, 0, abort_s);
    tc_fence_after();
    const bool warp_live = t0 + 32 * warp < a.T;   // warp-uniform: any of this warp's tokens exist
    if (ok && warp_live) {
      // TMEM -> registers -> this thread's row of a staging tile in the (now
      // idle) operand stages.  Rows are padded by 16 bytes so the eight threads
      // of a store phase hit different banks.
      const bool out_bf16 = kQuery || a.out_bf16;
      const uint32_t row_bytes = NT * (out_bf16 ? 2 : 4);
      const uint32_t srow = smem_u32(smem) + row * (row_bytes + 16);
      const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
      const bool live = t < a.T;
      auto stage_chunk = [&](int c, const uint32_t (&r)[32]) {
        if (!live) return;
        if (out_bf16) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_shared_v4(srow + 64 * c + 16 * i,
                         pack_bf16x2(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1])),
                         pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                         pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                         pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(srow + 128 * c + 16 * i, r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
        }
      };
      // 32 columns at a time; each load completes inside its own asm statement
      // (a load left in flight across other work could have its registers
      // copied before they are filled).
      uint32_t ra[32];
#pragma unroll 1
      for (int c = 0; c < NT / 32; ++c) {
        tmem_ld32_sync(lane_addr + 32 * c, ra);
        stage_chunk(c, ra);
      }
      // The warp then writes its own 32 staged rows out, one row segment per
      // coalesced store (16 bytes per lane).
      __syncwarp();
      const int64_t width = kQuery ? kDk : 128;
      const uint32_t esz = out_bf16 ? 2 : 4;
      const uint32_t lanes_per_row = row_bytes / 16;            // 32 or 16
      const int rows_per_iter = 32 / lanes_per_row;              // 1 or 2
      const int sub = lane / lanes_per_row, col16 = lane % lanes_per_row;
#pragma unroll 4
      for (int j = sub; j < 32; j += rows_per_iter) {
        const int rr = 32 * warp + j;
        const int64_t tt = t0 + rr;
        if (tt >= a.T) break;                                    // rows are in order: the rest are past T
        const uint4 x = ld_shared_v4(smem_u32(smem) + rr * (row_bytes + 16) + 16 * col16);
        uint8_t* g = reinterpret_cast<uint8_t*>(a.out) + ((tt * a.H + h) * width + n0) * esz + 16 * col16;
        *reinterpret_cast<uint4*>(g) = x;
      }
    }
  }

  if (*abort_s && tid == 0) flag(a.status, DCP_STATUS_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  // After an abort, let in-flight copies and products (microseconds) land
  // before the shared memory and TMEM are given back.
  if (*abort_s) __nanosleep(100000);
  tc_fence_after();
  if (warp == kIssuerWarp) tmem_dealloc(tmem, NT);
}

// ---------------------------------------------------------------------------- merge + output product
// The LSE merge of the N partials and the output-side product in one kernel
// ("MLA 的 Decode Context Parallelism", section 4, stage 7: the two-pass merge
// and the w_vc up-projection at the head owner): per head h and 16 query
// tokens (a work item), the merged latent output o[t, h, :] is formed in
// shared memory as a bf16 operand and multiplied by w_vc[h] on the tensor core;
// only v (and the merged lse) is written.  The merged o never reaches global
// memory.
// Persistent: at most one CTA per SM walks the work items (the grid is the
// fewest CTAs that still give each the largest share), its warps in six roles:
//   producers (warps 12 and 15, one thread each)  stream, two K-steps at a
//        time, each part's [16 tokens][128 dims] box of o_part by TMA into a
//        ring of shared-memory stages (144 KB in flight), and, on their own,
//        w_vc[h]'s [64 k][128 n] K-steps into a ring of two, so that neither
//        stream waits for the other's ring;
//   weights (warp 14)  the next item's row weights w_p = base^(lse_p - m) / Z
//        and merged lse, into one of two weight buffers, while the current
//        item is merged;
//   merge (warps 4-11)  reduce the parts stage by stage (sum_p w_p o_p, from
//        shared memory) and write each K-step's merged rows, rounded to bf16,
//        as a 128-byte-swizzled K-major B tile [16 tokens][64 k];
//   MMA (warp 13, one thread)  v^T = w_vc[h]^T o^T as soon as each tile is
//        written: A = w_vc[h] (MN-major, M = 128 output dims), B = the merged
//        tile (N = 16 tokens), K = 16 per product, into one of two TMEM
//        accumulators;
//   epilogue (warps 0-3)  TMEM lane = output dim, column = token: each token's
//        128 outputs go out as one coalesced row.
// Weights, B tiles and accumulators are double-buffered across items, so the
// merge warps stream without waiting for either end of an item.  HBM-bound:
// the partials (N * 512 * 4 bytes per row in f32) are read once; w_vc[h]
// (128 KB) once per item, mostly from L2.
constexpr int kMaThreads = 512;
constexpr int kMaMergeWarp0 = 4;
constexpr int kMaMergeWarps = 8;
constexpr int kMaProducerWarp = 12;
constexpr int kMaIssuerWarp = 13;
constexpr int kMaWeightsWarp = 14;
constexpr int kMaWProducerWarp = 15;
constexpr int kMaTok = 16;                    // query tokens per item (the product's N)
constexpr int kMaKSteps = kDv / kKStep;       // 8
constexpr int kMaBoxDims = 128;               // dims per o_part box (two K-steps; 256-dim boxes, half as
                                              // many stages, measured slower)
constexpr int kMaKPerBox = kMaBoxDims / kKStep;
constexpr int kMaWStages = 2;
constexpr int kMaMaxParts = 64;
constexpr uint32_t kMaRingBytes = 144 * 1024;                                // o_part stages
constexpr uint32_t kMaBTileBytes = kMaTok * 128;                             // [16 rows][64 k] bf16, 2 KB
constexpr uint32_t kMaWStageBytes = 2 * kWBoxBytes;                          // [64 k][128 n] bf16, 16 KB
constexpr uint32_t kMaRing = 0;
constexpr uint32_t kMaW = kMaRing + kMaRingBytes;                            // 2 W stages, 32 KB
constexpr uint32_t kMaB = kMaW + kMaWStages * kMaWStageBytes;                // 2 x 8 B tiles, 32 KB
constexpr uint32_t kMaWts = kMaB + 2 * kMaKSteps * kMaBTileBytes;            // weights [2][parts][16] f32, 8 KB
constexpr int kMaMaxStages = kMaRingBytes / (kMaTok * kMaBoxDims * 2);       // 36 (bf16 boxes)
// barriers: full[stages], empty[stages], w_full[2], w_empty[2], b_full[2][8], b_empty[2], d_full[2],
// d_empty[2], g_full[2], g_empty[2] (the weight buffers)
constexpr int kMaNumBars = 2 * kMaMaxStages + 2 * kMaWStages + 2 * kMaKSteps + 10;
constexpr uint32_t kMaBars = kMaWts + 2 * kMaMaxParts * kMaTok * 4;
constexpr uint32_t kMaMisc = kMaBars + kMaNumBars * 8;
constexpr uint32_t kMaBytes = kMaMisc + 16 + 1024;                            // + alignment slack

struct MergeAbsorbArgs {
  int64_t T;
  int32_t H, n_parts, base2;
  int32_t n_tiles, n_items;   // token tiles of 16, items = H * n_tiles
  const float* lse_part;      // [n_parts, T, H]
  void* v;                    // [T, H, 128] f32 or bf16
  int32_t v_bf16;
  float* lse;                 // [T, H] or null
  int32_t* status;
};

template <int kInBf16, int kBase2>
__global__ void __launch_bounds__(kMaThreads, 1)
    merge_absorb_kernel(const __grid_constant__ CUtensorMap tmap_o, const __grid_constant__ CUtensorMap tmap_w,
                        MergeAbsorbArgs a) {
  constexpr uint32_t kBoxBytes = kMaTok * kMaBoxDims * (kInBf16 ? 2 : 4);
  constexpr int kStages = kMaRingBytes / kBoxBytes;   // 18 (f32) or 36 (bf16)
  constexpr int kBoxesPerPart = kMaKSteps / kMaKPerBox;   // boxes per part and item
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* wts = reinterpret_cast<float*>(smem + kMaWts);  // [2][kMaMaxParts][16]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kMaBars);
  uint64_t* empty = full + kStages;
  uint64_t* w_full = empty + kStages;
  uint64_t* w_empty = w_full + kMaWStages;
  uint64_t* b_full = w_empty + kMaWStages;            // [2][8]
  uint64_t* b_empty = b_full + 2 * kMaKSteps;         // [2]
  uint64_t* d_full = b_empty + 2;                     // [2]
  uint64_t* d_empty = d_full + 2;                     // [2]
  uint64_t* g_full = d_empty + 2;                     // [2] weights ready
  uint64_t* g_empty = g_full + 2;                     // [2] weights no longer read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMaMisc);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + kMaMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.n_parts;

  if (warp == kMaProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_o);
    prefetch_tmap(&tmap_w);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMaMergeWarps);
    }
    for (int i = 0; i < kMaWStages; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 1);
    }
    for (int i = 0; i < 2 * kMaKSteps; ++i) mbar_init(&b_full[i], kMaMergeWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_empty[i], 1);
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);
      mbar_init(&g_full[i], 1);
      mbar_init(&g_empty[i], kMaMergeWarps);
    }
    *abort_s = 0;
    fence_barrier_init();
  }
  if (warp == kMaIssuerWarp) {
    tmem_alloc(tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kMaProducerWarp) {
    // ------------------------------------------------------------------ TMA producer: o_part boxes
    if (lane == 0) {
      uint32_t q = 0;  // o_part boxes issued so far
      bool ok = true;
      for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
        const int h = item / a.n_tiles;
        const int64_t t0 = (int64_t)(item % a.n_tiles) * kMaTok;
        for (int kb = 0; kb < kBoxesPerPart && ok; ++kb) {
          for (int p = 0; p < n && ok; ++p, ++q) {  // every part's [16 tokens][128 dims] box
            const uint32_t qs = q % kStages;
            if (!mbar_wait(&empty[qs], ((q / kStages) & 1) ^ 1, abort_s)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[qs], kBoxBytes);
            tma_load_3d(smem + kMaRing + qs * kBoxBytes, &tmap_o, &full[qs], kb * kMaBoxDims, h,
                        (int32_t)((int64_t)p * a.T + t0));
          }
        }
      }
    }
  } else if (warp == kMaWProducerWarp) {
    // ------------------------------------------------------------------ TMA producer: w_vc K-steps
    if (lane == 0) {
      uint32_t wq = 0;  // w_vc K-steps issued so far
      bool ok = true;
      for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
        const int h = item / a.n_tiles;
        for (int ks = 0; ks < kMaKSteps; ++ks, ++wq) {
          const uint32_t ws = wq % kMaWStages;
          if (!mbar_wait(&w_empty[ws], ((wq / kMaWStages) & 1) ^ 1, abort_s)) { ok = false; break; }
          uint8_t* st = smem + kMaW + ws * kMaWStageBytes;
          mbar_arrive_expect_tx(&w_full[ws], kMaWStageBytes);
          tma_load_3d(st, &tmap_w, &w_full[ws], 0, ks * kKStep, h);
          tma_load_3d(st + kWBoxBytes, &tmap_w, &w_full[ws], 64, ks * kKStep, h);
        }
      }
    }
  } else if (warp == kMaIssuerWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kMaTok, 1, 0);  // A = w_vc MN-major, B = o K-major
      uint32_t wq = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x, ++it) {
        const uint32_t buf = it & 1, use = (it >> 1) & 1;
        for (int ks = 0; ks < kMaKSteps && ok; ++ks, ++wq) {
          const uint32_t ws = wq % kMaWStages;
          if (!mbar_wait(&b_full[buf * kMaKSteps + ks], use, abort_s) ||
              !mbar_wait(&w_full[ws], (wq / kMaWStages) & 1, abort_s) ||
              (ks == 0 && !mbar_wait(&d_empty[buf], use ^ 1, abort_s))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t wdesc = sw128_desc(smem_u32(smem + kMaW + ws * kMaWStageBytes), kWBoxBytes, 1024);
          const uint64_t bdesc =
              sw128_desc(smem_u32(smem + kMaB + (buf * kMaKSteps + ks) * kMaBTileBytes), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kKStep / 16; ++kk)
            mma_bf16_ss(tmem + 16 * buf, wdesc + kk * (2048 >> 4), bdesc + kk * (32 >> 4), idesc, (ks | kk) != 0);
          mma_commit(&w_empty[ws]);
        }
        if (ok) {
          mma_commit(&d_full[buf]);
          mma_commit(&b_empty[buf]);
        }
      }
    }
  } else if (warp == kMaWeightsWarp) {
    // ------------------------------------------------------------------ row weights, one item ahead
    // lanes 0-15 serve the item's 16 tokens; every part's lse is loaded at once
    const int64_t rows = a.T * a.H;
    uint32_t it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x, ++it) {
      const int h = item / a.n_tiles;
      const int64_t t = (int64_t)(item % a.n_tiles) * kMaTok + (lane & 15);
      const uint32_t buf = it & 1, use = (it >> 1) & 1;
      if (!warp_wait_all(&g_empty[buf], use ^ 1, abort_s)) { ok = false; break; }
      float* w = wts + buf * kMaMaxParts * kMaTok;
      if (lane < kMaTok) {
        const bool live = t < a.T;
        float m = -INFINITY;
        for (int p = 0; p < n; ++p) {
          const float l = live ? __ldg(a.lse_part + p * rows + t * a.H + h) : -INFINITY;
          w[p * kMaTok + lane] = l;
          m = fmaxf(m, l);
        }
        float z = 0.f;
        for (int p = 0; p < n; ++p) {
          const float l = w[p * kMaTok + lane];
          const float e = (m == -INFINITY || l == -INFINITY) ? 0.f : (kBase2 ? exp2f(l - m) : expf(l - m));
          w[p * kMaTok + lane] = e;
          z += e;
        }
        const float inv = z > 0.f ? 1.f / z : 0.f;
        for (int p = 0; p < n; ++p) w[p * kMaTok + lane] *= inv;
        if (live && a.lse) a.lse[t * a.H + h] = z > 0.f ? m + (kBase2 ? log2f(z) : logf(z)) : -INFINITY;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&g_full[buf]);
    }
  } else if (warp >= kMaMergeWarp0) {
    // ------------------------------------------------------------------ merge warps 4-11
    const int mt = tid - 32 * kMaMergeWarp0;  // 0 .. 255
    const int r = mt >> 4;                    // this thread's token within the item
    const int c4 = mt & 15;                   // its 4-dim group within each 64-dim K-step
    uint32_t q = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x, ++it) {
      const uint32_t buf = it & 1, use = (it >> 1) & 1;
      // the item's weights, and this buffer's B tiles free (products of two items ago done)
      if (!warp_wait_all(&g_full[buf], use, abort_s) || !warp_wait_all(&b_empty[buf], use ^ 1, abort_s)) {
        ok = false;
        break;
      }
      const float* w = wts + buf * kMaMaxParts * kMaTok;
      for (int kb = 0; kb < kBoxesPerPart && ok; ++kb) {
        float4 acc[kMaKPerBox];
#pragma unroll
        for (int j = 0; j < kMaKPerBox; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < n; ++p, ++q) {
          const uint32_t qs = q % kStages;
          if (!warp_wait_all(&full[qs], (q / kStages) & 1, abort_s)) { ok = false; break; }
          const float wp = w[p * kMaTok + r];
          const uint8_t* box = smem + kMaRing + qs * kBoxBytes;
          float4 x[kMaKPerBox];  // dims [64 j + 4 c4, +4) of K-step j of the box
#pragma unroll
          for (int j = 0; j < kMaKPerBox; ++j) {
            if (kInBf16) {
              const uint2 u = *reinterpret_cast<const uint2*>(box + r * kMaBoxDims * 2 + j * 128 + c4 * 8);
              const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
              const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
              x[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
              x[j] = *reinterpret_cast<const float4*>(box + r * kMaBoxDims * 4 + j * 256 + c4 * 16);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[qs]);
#pragma unroll
          for (int j = 0; j < kMaKPerBox; ++j) {
            acc[j].x = fmaf(wp, x[j].x, acc[j].x); acc[j].y = fmaf(wp, x[j].y, acc[j].y);
            acc[j].z = fmaf(wp, x[j].z, acc[j].z); acc[j].w = fmaf(wp, x[j].w, acc[j].w);
          }
        }
        if (!ok) break;
        // the box's K-steps of the merged rows -> bf16, swizzled K-major:
        // 16-byte chunk c16 of row r at r * 128 + ((c16 ^ (r % 8)) * 16)
#pragma unroll
        for (int j = 0; j < kMaKPerBox; ++j) {
          const uint32_t off = kMaB + (buf * kMaKSteps + kMaKPerBox * kb + j) * kMaBTileBytes + r * 128 +
                               ((((c4 >> 1) ^ (r & 7))) << 4) + (c4 & 1) * 8;
          st_shared_v2(smem_u32(smem) + off, pack_bf16x2(acc[j].x, acc[j].y), pack_bf16x2(acc[j].z, acc[j].w));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < kMaKPerBox; ++j) mbar_arrive(&b_full[buf * kMaKSteps + kMaKPerBox * kb + j]);
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&g_empty[buf]);  // this item's weights are no longer read
    }
  } else {
    // ------------------------------------------------------------------ epilogue warps 0-3
    // TMEM lane 32w + l holds output dim 32w + l for the item's 16 tokens
    // (columns).  The TMEM load is warp-collective (.sync.aligned): every lane
    // runs it; only the stores depend on the token being live.
    uint32_t it = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++it) {
      const int h = item / a.n_tiles;
      const int64_t t0 = (int64_t)(item % a.n_tiles) * kMaTok;
      const uint32_t buf = it & 1, use = (it >> 1) & 1;
      if (!warp_wait_all(&d_full[buf], use, abort_s)) break;
      tc_fence_after();
      uint32_t rv[16];
      tmem_ld32x16_sync(tmem + ((uint32_t)(32 * warp) << 16) + 16 * buf, rv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[buf]);
      const int nd = 32 * warp + lane;
#pragma unroll
      for (int j = 0; j < kMaTok; ++j) {
        const int64_t t = t0 + j;
        if (t >= a.T) break;
        if (a.v_bf16)
          static_cast<__nv_bfloat16*>(a.v)[(t * a.H + h) * 128 + nd] = __float2bfloat16_rn(__uint_as_float(rv[j]));
        else
          static_cast<float*>(a.v)[(t * a.H + h) * 128 + nd] = __uint_as_float(rv[j]);
      }
    }
  }

  if (*abort_s && tid == 0) flag(a.status, DCP_STATUS_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (*abort_s) __nanosleep(100000);
  tc_fence_after();
  if (warp == kMaIssuerWarp) tmem_dealloc(tmem, 32);
}

// bf16 A rows of K elements: dims (k, head, token), box [128 tokens][1][64 k].
bool make_tmap_a(CUtensorMap* m, const void* base, int64_t K, int64_t H, int64_t T, int64_t row_stride) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)row_stride * H * 2};
  cuuint32_t box[3] = {(cuuint32_t)kKStep, 1, (cuuint32_t)kTokTile};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 weights [H, K, N] (N innermost): box [1][64 k][64 n].
bool make_tmap_w(CUtensorMap* m, const void* base, int64_t H, int64_t K, int64_t N) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)K, (cuuint64_t)H};
  cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)K * N * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kKStep, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Raise the kernel's dynamic shared-memory limit, once per instance and device.
template <int NT, int KSTEPS, int STAGES, bool kQuery, bool kAF32>
bool prepare() {
  static SmemLimit limit;
  return limit.ensure(reinterpret_cast<const void*>(&absorb_kernel<NT, KSTEPS, STAGES, kQuery, kAF32>),
                      AbsorbSmem<NT, KSTEPS, STAGES>::kBytes);
}

template <int NT, int KSTEPS, int STAGES, bool kQuery, bool kAF32>
int32_t launch(const CUtensorMap& ta, const CUtensorMap& tw, const AbsorbArgs& a, int n_tiles, cudaStream_t st) {
  if (!prepare<NT, KSTEPS, STAGES, kQuery, kAF32>()) return DCP_ERR_CUDA;
  const dim3 grid((unsigned)n_tiles, (unsigned)a.H, (unsigned)((a.T + kTokTile - 1) / kTokTile));
  absorb_kernel<NT, KSTEPS, STAGES, kQuery, kAF32>
      <<<grid, kAbsThreads, AbsorbSmem<NT, KSTEPS, STAGES>::kBytes, st>>>(ta, tw, a);
  return launch_status();
}

bool sizes_ok(int64_t T, int32_t H) {
  return T >= 0 && H >= 1 && H <= 65535 && (T + kTokTile - 1) / kTokTile <= 65535;
}

}  // namespace

extern "C" int32_t dcp_absorb_q(int64_t T, int32_t H, const void* q_nope, int64_t q_nope_stride, const void* q_pe,
                                int64_t q_pe_stride, const void* w_kc, void* q, int32_t* status, void* stream) {
  if (!sizes_ok(T, H)) return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!q_nope || !q_pe || !w_kc || !q) return DCP_ERR_INVALID;
  if (q_nope_stride < 128 || q_nope_stride % 8 || q_pe_stride < 64 || q_pe_stride % 8) return DCP_ERR_INVALID;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(w_kc) || !aligned16(q)) return DCP_ERR_INVALID;
  CUtensorMap ta, tw;
  if (!make_tmap_a(&ta, q_nope, 128, H, T, q_nope_stride) || !make_tmap_w(&tw, w_kc, H, 128, kDv))
    return DCP_ERR_CUDA;
  AbsorbArgs a{};
  a.T = T;
  a.H = H;
  a.out = q;
  a.out_bf16 = 1;
  a.q_pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  a.q_pe_stride = q_pe_stride;
  a.status = status;
  return launch<kQTile, 2, 2, true, false>(ta, tw, a, kDv / kQTile, as_stream(stream));
}

extern "C" int32_t dcp_absorb_o(int64_t T, int32_t H, const void* o, int32_t o_dtype, const void* w_vc, void* v,
                                int32_t v_dtype, int32_t* status, void* stream) {
  if (!sizes_ok(T, H)) return DCP_ERR_INVALID;
  if ((o_dtype != DCP_F32 && o_dtype != DCP_BF16) || (v_dtype != DCP_F32 && v_dtype != DCP_BF16))
    return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!o || !w_vc || !v) return DCP_ERR_INVALID;
  if (!aligned16(o) || !aligned16(w_vc) || !aligned16(v)) return DCP_ERR_INVALID;
  CUtensorMap ta, tw;
  if (!make_tmap_w(&tw, w_vc, H, kDv, 128)) return DCP_ERR_CUDA;
  AbsorbArgs a{};
  a.T = T;
  a.H = H;
  a.out = v;
  a.out_bf16 = v_dtype == DCP_BF16;
  a.status = status;
  if (o_dtype == DCP_BF16) {
    if (!make_tmap_a(&ta, o, kDv, H, T, kDv)) return DCP_ERR_CUDA;
    return launch<kOTile, 8, kOStages, false, false>(ta, tw, a, 128 / kOTile, as_stream(stream));
  }
  a.a_f32 = reinterpret_cast<const float*>(o);
  a.a_f32_stride = kDv;
  return launch<kOTile, 8, kOStages, false, true>(tw, tw, a, 128 / kOTile, as_stream(stream));
}

namespace {

template <int kInBf16, int kBase2>
int32_t launch_merge_absorb(const CUtensorMap& to, const CUtensorMap& tw, const MergeAbsorbArgs& a, cudaStream_t st) {
  static SmemLimit limit;
  if (!limit.ensure(reinterpret_cast<const void*>(&merge_absorb_kernel<kInBf16, kBase2>), kMaBytes))
    return DCP_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return DCP_ERR_CUDA;
  // persistent, at most one CTA per SM: the fewest CTAs that still give each the
  // same largest share of items (384 items on 152 SMs: 128 CTAs of 3, not 152
  // CTAs of 2 or 3), so that no SM's bandwidth goes to a short share
  const int per_cta = (a.n_items + sms - 1) / sms;
  const int grid = (a.n_items + per_cta - 1) / per_cta;
  merge_absorb_kernel<kInBf16, kBase2><<<grid, kMaThreads, kMaBytes, st>>>(to, tw, a);
  return launch_status();
}

// o_part [n_parts, T, H, 512] seen as (dims, head, part-major token row):
// boxes of [16 rows][1 head][128 dims], no swizzle.
bool make_tmap_parts(CUtensorMap* m, const void* base, int n_parts, int64_t T, int64_t H, bool bf16) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  const uint64_t e = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)kDv, (cuuint64_t)H, (cuuint64_t)(n_parts * T)};
  cuuint64_t strides[2] = {(cuuint64_t)kDv * e, (cuuint64_t)(H * kDv * e)};
  cuuint32_t box[3] = {(cuuint32_t)kMaBoxDims, 1, (cuuint32_t)kMaTok};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int32_t dcp_lse_merge_absorb_o(int32_t n_parts, int64_t T, int32_t H, const void* o_part,
                                          int32_t o_part_dtype, const float* lse_part, int32_t lse_base,
                                          const void* w_vc, void* v, int32_t v_dtype, float* lse, int32_t* status,
                                          void* stream) {
  if (n_parts < 1 || n_parts > kMaMaxParts || T < 0 || H < 1 || H > 65535) return DCP_ERR_INVALID;
  if ((o_part_dtype != DCP_F32 && o_part_dtype != DCP_BF16) || (v_dtype != DCP_F32 && v_dtype != DCP_BF16))
    return DCP_ERR_INVALID;
  if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2) return DCP_ERR_INVALID;
  if (T == 0) return DCP_OK;
  if (!o_part || !lse_part || !w_vc || !v) return DCP_ERR_INVALID;
  if (!aligned16(o_part) || !aligned16(w_vc) || !aligned16(v)) return DCP_ERR_INVALID;
  const int64_t n_tiles = (T + kMaTok - 1) / kMaTok;
  if (n_tiles * H > INT32_MAX || (int64_t)n_parts * T > INT32_MAX) return DCP_ERR_UNSUPPORTED;
  const bool ib = o_part_dtype == DCP_BF16;
  CUtensorMap to, tw;
  if (!make_tmap_parts(&to, o_part, n_parts, T, H, ib) || !make_tmap_w(&tw, w_vc, H, kDv, 128)) return DCP_ERR_CUDA;
  MergeAbsorbArgs a{};
  a.T = T;
  a.H = H;
  a.n_parts = n_parts;
  a.base2 = lse_base == DCP_LSE_BASE_2;
  a.n_tiles = (int32_t)n_tiles;
  a.n_items = (int32_t)(n_tiles * H);
  a.lse_part = lse_part;
  a.v = v;
  a.v_bf16 = v_dtype == DCP_BF16;
  a.lse = lse;
  a.status = status;
  cudaStream_t st = as_stream(stream);
  if (ib) return a.base2 ? launch_merge_absorb<1, 1>(to, tw, a, st) : launch_merge_absorb<1, 0>(to, tw, a, st);
  return a.base2 ? launch_merge_absorb<0, 1>(to, tw, a, st) : launch_merge_absorb<0, 0>(to, tw, a, st);
}
