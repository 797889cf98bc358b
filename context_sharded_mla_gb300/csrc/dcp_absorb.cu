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
