/*
 * dcp.h — C ABI of the sharded absorbed-MLA decode library (sm_103a / GB300).
 *
 * The library implements the data-parallel hot path of Decode Context
 * Parallelism (DCP) for absorbed Multi-head Latent Attention:
 *
 *   1. dcp_slot_map            owner / local row / physical slot of each new token
 *   2. dcp_kv_append           owner-filtered write of the 576-d latent rows
 *   3. dcp_mla_decode_partial  per-shard partial attention (o_r, lse_r)
 *   4. dcp_lse_merge           exact log-sum-exp merge of the N partials
 * and, for moving a request prefilled without context sharding into the shards,
 *   5. dcp_kv_relayout         owner-filtered copy from a paged prefill pool
 * and, on either side of the attention, the two absorption products
 *   6. dcp_absorb_q            q_nope @ w_kc -> the 576-d absorbed query
 *   7. dcp_absorb_o            merged latent output @ w_vc -> per-head value
 *      dcp_lse_merge_absorb_o  the merge and that product in one kernel
 * and, when the shards are spread over W GPUs (one rank each), the two sides
 * of the exchange of the partials
 *   8. dcp_pack_partials       head slice d of every held shard -> rank d's chunk
 *   9. dcp_lse_merge_packed    the head owner's merge, read from its receive buffer
 *  10. dcp_lse_rescale         the local step of the AllGather + ReduceScatter form
 *
 * On one GPU the N context shards are N compact paged pools in one HBM
 * allocation (the "arena"), so the cross-rank steps (query all-gather,
 * all-to-all of the partials) become plain device buffers.  Over W GPUs each
 * holds N / W consecutive shards; the caller runs the collective itself
 * (e.g. NCCL all-to-all) between dcp_pack_partials and dcp_lse_merge_packed.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All pointers except `layout` and the host scalars are DEVICE pointers
 *    (CUDA global memory of the current device).  The caller allocates and
 *    frees every buffer; no call allocates device memory or keeps state
 *    between calls.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls only enqueue work; they do not synchronise.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns DCP_ERR_INVALID (or DCP_ERR_UNSUPPORTED) and launches
 *    nothing.  A failed launch returns DCP_ERR_CUDA.
 *  - Data-dependent range errors found on the device (a negative position, a
 *    local row past the block table, a page id outside the pool, a sequence
 *    length the block table cannot hold) OR a DCP_STATUS_* bit into the
 *    caller's device word `*status` and skip the offending read or write.
 *    `status` is sticky: the library never clears it.  No kernel traps.
 *  - bf16 means IEEE bfloat16 stored as 16-bit words; f32 is IEEE binary32.
 *  - Tensors are dense and row-major ("C order") in the shapes given.
 *
 * Notation: N = layout->n_shards, I = layout->interleave (1 = token
 * round-robin), P = layout->page_size (rows per physical page), Dk = 576
 * latent dims (512 c_K + 64 k_R), Dv = 512 value dims (the c_K part).
 */
#ifndef DCP_H_
#define DCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shard layout.  Source: "PCP / DCP：计算、KV 布局与块轮转", section 6 (block
 * round-robin with block size B, here `interleave`), and vLLM-Ascend
 * "上下文并行（CP）", section "块表" (cp_kv_cache_interleave_size; the page size
 * must be a multiple of it).  Requirements: n_shards >= 1, interleave >= 1,
 * page_size >= 1 and page_size % interleave == 0. */
typedef struct dcp_layout {
  int32_t n_shards;
  int32_t interleave;
  int32_t page_size;
} dcp_layout_t;

/* Return codes. */
enum {
  DCP_OK = 0,
  DCP_ERR_INVALID = -1,      /* bad argument (null pointer, size, layout, dtype) */
  DCP_ERR_UNSUPPORTED = -2,  /* valid but outside what this build handles */
  DCP_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed */
  DCP_ERR_WORKSPACE = -4,    /* workspace missing or smaller than required */
  DCP_ERR_TOO_LARGE = -5     /* sizes need more scratch than the library's built-in area */
};

/* Device status bits (OR-ed into *status). */
enum {
  DCP_STATUS_BAD_POSITION = 1,    /* position < 0 */
  DCP_STATUS_BAD_PAGE_INDEX = 2,  /* local row / P >= max_pages */
  DCP_STATUS_BAD_PAGE_ID = 4,     /* block-table entry outside [0, pool_pages) */
  DCP_STATUS_BAD_REQUEST = 8,     /* request index outside [0, B) */
  DCP_STATUS_BAD_LENGTH = 16,     /* seq_len < q_len */
  DCP_STATUS_TIMEOUT = 32,        /* a kernel pipeline wait gave up (the call's outputs are invalid) */
  DCP_STATUS_INTERNAL = 64        /* a kernel found its shared memory misaligned and did nothing (outputs invalid) */
};

enum { DCP_LSE_BASE_E = 0, DCP_LSE_BASE_2 = 1 };
enum { DCP_F32 = 0, DCP_BF16 = 1 };

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t dcp_version(void);

/* Short English description of a return code (static storage). */
const char* dcp_error_string(int32_t code);

/* Number of CUDA kernels this library has launched in this process so far
 * (all entry points, all devices).  Host-only; lets a caller count the
 * library's launches inside a timed region. */
int64_t dcp_launch_count(void);

/*
 * dcp_count — number of positions p in [0, x) owned by `shard`; host-only, pure.
 *
 * Source: "Decode Context Parallelism" (zdszero), section "Core abstraction",
 * idea 1 (a chunk [a, a+L) gives a shard count(a+L) - count(a) positions), and
 * "PCP / DCP：计算、KV 布局与块轮转", section 6, local_len:
 *   count(x) = (x / (N*I)) * I + clamp(x % (N*I) - shard*I, 0, I).
 * Returns -1 on a bad layout, shard outside [0, N) or x < 0.
 */
int64_t dcp_count(const dcp_layout_t* layout, int32_t shard, int64_t x);

/*
 * dcp_slot_map — placement of T new tokens.
 *
 * Sources: "Decode Context Parallelism" (zdszero), "Core abstraction" idea 1
 * (owner(p) = p mod N, row(p) = floor(p / N)); "PCP / DCP：计算、KV 布局与块轮转"
 * section 6 (owner = (p / I) % N, local row = (p / (N*I)) * I + p % I) and
 * section "KV cache 管理" (slot = page_id * P + offset_in_page); SGLang
 * "Decode context parallelism", "Virtual KV layout" (one shared block table;
 * a widened page of N*P positions maps to one physical page on every shard).
 *
 *   pos          int64[T]  request-global positions (>= 0)
 *   req          int32[T]  request index of each token, in [0, B)
 *   block_table  int32[B, bt_stride]; entry [b][k] is the physical page (same
 *                id on every shard) holding local rows [k*P, (k+1)*P) of b;
 *                only columns k < max_pages are read
 *   B            rows of block_table: a token whose request lies outside [0, B)
 *                is flagged (BAD_REQUEST) instead of read past the table
 *   pool_pages   pages per shard pool: a page id outside [0, pool_pages) gives
 *                slot -1 and BAD_PAGE_ID, so no caller writes past a pool
 *   owner  (out) int32[T]  owning shard
 *   row    (out) int64[T]  local row on the owner
 *   slot   (out) int64[T]  row index inside the owner's pool = page * P + row % P,
 *                          or -1 if the token could not be placed (status set)
 *   status (in/out) int32 device word, see DCP_STATUS_*
 * T == 0 is a no-op.  Errors: DCP_ERR_INVALID for a bad layout, T < 0,
 * B < 1, max_pages < 1 or max_pages > bt_stride, pool_pages < 1, or a null
 * pointer with T > 0.
 */
int32_t dcp_slot_map(const dcp_layout_t* layout, const int64_t* pos, const int32_t* req,
                     int64_t T, const int32_t* block_table, int32_t B, int64_t bt_stride,
                     int64_t max_pages, int64_t pool_pages, int32_t* owner, int64_t* row,
                     int64_t* slot, int32_t* status, void* stream);

/*
 * dcp_kv_append — owner-filtered write of new latent rows.
 *
 * Source: "MLA 的 Decode Context Parallelism", section 4, stage 2 (every rank
 * computes the new latent [c_K || k_R]; only the owner stores its row) and
 * section 6 (set_mla_kv_buffer_dcp_sharded); "Decode Context Parallelism"
 * (zdszero), SGLang K3 decode path (the new token's latent is written only to
 * its owner rank).  Placement is dcp_slot_map's, computed in the same kernel.
 *
 *   kv_new       bf16[T, 576]  new latent rows
 *   pos, req     int64[T], int32[T]: request-global position and request index
 *                of each new token (as for dcp_slot_map)
 *   block_table  int32[B, bt_stride], columns k < max_pages read (as for
 *                dcp_slot_map)
 *   arena        bf16[shard_end - shard_begin, pool_pages * P, 576]: the pools
 *                of shards [shard_begin, shard_end), one after another
 * Token t with owner o = (pos / I) % N in [shard_begin, shard_end) is copied bit
 * for bit to arena[o - shard_begin][slot], slot = block_table[req][row / P] * P
 * + row % P with row = (pos / (N*I)) * I + pos % I; tokens of other shards are
 * skipped (another device holds them) and their block-table entries are not
 * read.  Device status: a negative position (BAD_POSITION) or a request outside
 * [0, B) (BAD_REQUEST) is flagged for any token; a local row past max_pages
 * (BAD_PAGE_INDEX) or a page id outside [0, pool_pages) (BAD_PAGE_ID) for a
 * held token; each skips only that token.  T == 0 is a no-op.  Errors:
 * DCP_ERR_INVALID for a bad layout or shard range, T < 0, B < 1, max_pages
 * outside [1, bt_stride], pool_pages < 1, a null pointer with T > 0, or kv_new
 * / arena not 16-byte aligned.
 */
int32_t dcp_kv_append(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                      const void* kv_new, const int64_t* pos, const int32_t* req, int64_t T,
                      const int32_t* block_table, int32_t B, int64_t bt_stride, int64_t max_pages,
                      void* arena, int64_t pool_pages, int32_t* status, void* stream);

/*
 * dcp_kv_relayout — prefill-to-decode relayout of latent rows into the shards.
 *
 * Source: "PCP / DCP：计算、KV 布局与块轮转", section "PD + DCP：从完整源页
 * 抽取本 rank 的 token" (a request prefilled without context sharding, in full
 * pages, moves to a DCP decode instance: each rank keeps the tokens whose
 * request position it owns -- chosen by position, not by physical slot --
 * reads them from their source slots and writes them compactly into its own
 * pages) and section "Block RR 改善哪一段" (with block round-robin whole
 * contiguous pages move).
 *
 *   src_pool         bf16[src_pool_rows, 576]  the prefill side's paged pool
 *   src_block_table  int32[B, src_bt_stride]; entry [b][k] is the source page
 *                    holding request positions [k*src_page_size, (k+1)*src_page_size)
 *                    of b; only columns k < src_max_pages are read
 *   pos, req         int64[T], int32[T]: the request position and request of
 *                    each token to move (e.g. positions [a, a+L) of a chunk)
 *   block_table, arena, pool_pages: the decode side, as in dcp_slot_map and
 *                    dcp_kv_append (arena holds shards [shard_begin, shard_end))
 * Token t with owner(pos[t]) in [shard_begin, shard_end) is copied bit for bit
 * from src_pool[src_block_table[req][pos / src_page_size] * src_page_size +
 * pos % src_page_size] to arena[owner - shard_begin][slot], slot as in
 * dcp_slot_map; tokens of other shards are neither read nor written.  A
 * negative position, a request outside [0, B), a page index past max_pages /
 * src_max_pages, or a page id whose rows fall outside the pool (source or
 * destination) sets the DCP_STATUS_* bit and skips that token.  src_pool and
 * arena must not overlap.  T == 0 is a no-op.  Errors: DCP_ERR_INVALID for a
 * bad layout or shard range, T < 0, B < 1, src_page_size < 1, max_pages or
 * src_max_pages outside [1, stride], pool sizes < 1, a null pointer with T > 0,
 * or src_pool / arena not 16-byte aligned.
 */
int32_t dcp_kv_relayout(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                        const void* src_pool, int64_t src_pool_rows, int32_t src_page_size,
                        const int32_t* src_block_table, int64_t src_bt_stride, int64_t src_max_pages,
                        const int64_t* pos, const int32_t* req, int64_t T, int32_t B,
                        const int32_t* block_table, int64_t bt_stride, int64_t max_pages, void* arena,
                        int64_t pool_pages, int32_t* status, void* stream);

/*
 * dcp_mla_decode_partial — locally normalised partial attention of each shard.
 *
 * Sources: "MLA 的 Decode Context Parallelism", section 2 (absorbed form:
 * 576-d single-KV-head MQA, query per head [q_hat_C || q_R], value = c_K, the
 * first 512 dims of the latent row) and section 3 (each rank returns o^(r) and
 * lse_r); "Decode Context Parallelism" (zdszero), "Core abstraction" idea 2
 * (O_r = softmax_local(q k^T * scale) V_r, L_r = log sum_{p in P_r} exp(s_p));
 * "PCP / DCP：计算、KV 布局与块轮转" section 4.1 (an empty shard contributes a
 * zero-weight state); SGLang "Decode context parallelism", "DCP x speculative
 * decoding" (the verify kernel sees the shard rank and the GLOBAL lengths so the
 * causal mask spans the whole sequence).
 *
 * For request b with S_b = seq_lens[b] cached tokens (the q_len new ones
 * included), query token t sits at position S_b - q_len + t and sees every
 * position p <= S_b - q_len + t.  For each held shard r, query token t and
 * head h, with V_r the visible positions owned by r:
 *   s_p     = scale * sum_{d<576} q[b,t,h,d] * k_p[d]
 *   lse_r   = ln sum_{p in V_r} exp(s_p)      (log2 of the same sum if lse_base == 1)
 *   o_r     = sum_{p in V_r} exp(s_p - lse_e) * k_p[0:512]
 *   V_r empty -> lse_r = -inf, o_r = 0.
 *
 *   q          bf16[B, q_len, H, 576]
 *   arena      bf16[shard_end - shard_begin, pool_pages * P, 576]
 *   block_table, bt_stride, max_pages: as for dcp_slot_map
 *   seq_lens   int64[B] (device)
 *   o_part     [shard_end - shard_begin, B, q_len, H, 512], f32 or bf16 (o_part_dtype)
 *   lse_part   f32[shard_end - shard_begin, B, q_len, H]
 *   workspace  device scratch of at least dcp_mla_decode_workspace_size(...)
 *              bytes, 256-byte aligned; its contents need not be initialised
 *              and are meaningless after the call
 * Rows of a page past the request's length are read but carry zero weight;
 * they must hold finite values (a zero-initialised pool and dcp_kv_append
 * guarantee that).  Supported: 1 <= H, q_len * H <= 65536, B >= 1.  A large
 * q_len is a chunked extend in the all-gather-Q form: the chunk's query tokens
 * attend to every shard's rows exactly as decode tokens do, causally in global
 * positions (vLLM-Ascend "上下文并行（CP）", chunked prefill: the work after
 * gathering Q is the decode work).
 * Errors: DCP_ERR_INVALID on bad sizes/pointers/dtype/base, DCP_ERR_WORKSPACE
 * if the workspace is too small.  Device status: BAD_LENGTH, BAD_PAGE_ID.
 */
int32_t dcp_mla_decode_partial(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                               const void* q, int32_t B, int32_t q_len, int32_t H,
                               const void* arena, int64_t pool_pages,
                               const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                               const int64_t* seq_lens, float scale, int32_t lse_base,
                               void* o_part, int32_t o_part_dtype, float* lse_part,
                               void* workspace, size_t workspace_bytes,
                               int32_t* status, void* stream);

/* Workspace bytes dcp_mla_decode_partial needs for these sizes on the current
 * device (0 on bad arguments).  It does not depend on the sequence lengths (so
 * no maximum length is asked for); it depends on the number of shards held,
 * shard_end - shard_begin, through the (request, shard) work units. */
size_t dcp_mla_decode_workspace_size(const dcp_layout_t* layout, int32_t shard_begin,
                                     int32_t shard_end, int32_t B, int32_t q_len, int32_t H);

/*
 * dcp_lse_merge — exact merge of n_parts partials per row.
 *
 * Sources: "Decode Context Parallelism" (zdszero), "Theory": merge identity
 * O = sum_r exp(L_r) O_r / sum_r exp(L_r), its stable form with m = max_r L_r,
 * L = m + log sum_r exp(L_r - m), and the rule that exp/log must match the
 * base the kernel reported; "MLA 的 Decode Context Parallelism", section 3
 * (w_r = exp2(lse_r - m), out = sum_r w_r o^(r) / sum_r w_r); SGLang "Decode
 * context parallelism", "MLA decode dataflow" (lse = logsumexp_r lse_r,
 * o = sum_r exp(lse_r - lse) o_r, base e or base 2).
 *
 *   o_part   [n_parts, rows, 512] f32 or bf16 (o_part_dtype)
 *   lse_part f32[n_parts, rows], in base e (lse_base 0) or base 2 (lse_base 1)
 *   o        [rows, 512] f32 or bf16 (o_dtype)
 *   lse      f32[rows] in the same base (may be NULL if not wanted)
 * A part with lse = -inf has zero weight; a row whose parts are all -inf gets
 * o = 0 and lse = -inf.  rows == 0 is a no-op.  Errors: DCP_ERR_INVALID.
 */
int32_t dcp_lse_merge(int32_t n_parts, int64_t rows, const void* o_part, int32_t o_part_dtype,
                      const float* lse_part, int32_t lse_base, void* o, int32_t o_dtype,
                      float* lse, void* stream);

/*
 * dcp_mla_decode_partial_static — dcp_mla_decode_partial without a caller workspace.
 *
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory for a workspace — a serving process that has given all
 * free HBM to its KV pool and allows no further allocations, or a plain C host
 * program with no device-memory manager.  It computes exactly what
 * dcp_mla_decode_partial computes, with the same arguments minus the workspace,
 * and allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * Scratch comes from a file-scope device array of
 * dcp_mla_decode_static_scratch_bytes() bytes (64 MiB) that every GPU holds from
 * the moment it loads this library until the process exits.  The first call on
 * a device looks up that array's device address (cudaGetSymbolAddress, with the
 * device current); make that first call before any stream capture.  Every call
 * on a device shares the one array and leaves its contents behind; nothing in it
 * has to start at zero.  Calls whose work overlaps on the GPU (different streams,
 * or different host threads without ordering) race on the array and give wrong
 * results: order them.
 * Errors: as dcp_mla_decode_partial, plus DCP_ERR_TOO_LARGE when
 * dcp_mla_decode_workspace_size(...) for these sizes exceeds the array.
 */
int32_t dcp_mla_decode_partial_static(const dcp_layout_t* layout, int32_t shard_begin, int32_t shard_end,
                                      const void* q, int32_t B, int32_t q_len, int32_t H,
                                      const void* arena, int64_t pool_pages,
                                      const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                                      const int64_t* seq_lens, float scale, int32_t lse_base,
                                      void* o_part, int32_t o_part_dtype, float* lse_part,
                                      int32_t* status, void* stream);

/* Size in bytes of the built-in scratch array dcp_mla_decode_partial_static uses. */
size_t dcp_mla_decode_static_scratch_bytes(void);

/*
 * dcp_absorb_q — the query-side absorption product (identity 1).
 *
 * Sources: "MLA 的 Decode Context Parallelism", section 2 (identity 1: the K
 * up-projection moves into the query, q_hat_h = q^C W^UK_h in R^512, and the
 * decode query of head h is [q_hat_h || q^R_h], 576 dims); "Decode Context
 * Parallelism" (zdszero), section "decode 路径：以 Kimi K3 的 MLA 为例"
 * (w_kc [H, 128, 512] from the K part of kv_b_proj; bmm(q_nope, w_kc) ->
 * [B, H, 512]; q_pe enters attention unrotated).
 *
 *   T            query tokens (B x q_len; row t = b * q_len + i)
 *   q_nope       bf16, row (t, h) at element (t * H + h) * q_nope_stride; its
 *                first 128 elements are read.  q_nope_stride >= 128 and a
 *                multiple of 8 (a q_b_proj output [T, H, 192] passes its base
 *                with stride 192).
 *   q_pe         bf16, row (t, h) at (t * H + h) * q_pe_stride; 64 elements
 *                read; q_pe_stride >= 64, a multiple of 8.
 *   w_kc         bf16 [H, 128, 512]
 *   q     (out)  bf16 [T, H, 576]: dims [0, 512) = q_nope[t, h] @ w_kc[h]
 *                (f32 accumulation, rounded to nearest bf16), dims [512, 576)
 *                = q_pe[t, h] unchanged.  This is the `q` operand of
 *                dcp_mla_decode_partial.  Must not overlap the inputs.
 *   status       device word (may be NULL); DCP_STATUS_TIMEOUT if a pipeline
 *                wait gave up (q is then invalid).
 * Every pointer must be 16-byte aligned.  T == 0 is a no-op.  Errors:
 * DCP_ERR_INVALID on T < 0, H < 1 or H > 65535, more than 65535 tiles of 128
 * tokens, a null or misaligned pointer, or a bad stride.
 */
int32_t dcp_absorb_q(int64_t T, int32_t H, const void* q_nope, int64_t q_nope_stride, const void* q_pe,
                     int64_t q_pe_stride, const void* w_kc, void* q, int32_t* status, void* stream);

/*
 * dcp_absorb_o — the output-side absorption product (identity 2).
 *
 * Sources: "MLA 的 Decode Context Parallelism", section 2 (identity 2: the
 * attention-weighted sum of W^UV_h c_t equals W^UV_h applied once to the
 * weighted sum of latent rows); "Decode Context Parallelism" (zdszero),
 * section "decode 路径：以 Kimi K3 的 MLA 为例" (w_vc [H, 512, 128] from the
 * V part of kv_b_proj; bmm(O, w_vc) -> [B, H, 128] after the merge).
 *
 *   o            [T, H, 512] f32 or bf16 (o_dtype): the merged latent output
 *                (dcp_lse_merge's `o` with rows = T * H).  An f32 o is rounded
 *                to nearest bf16 in the kernel before the product (the tensor
 *                core multiplies bf16 by bf16).
 *   w_vc         bf16 [H, 512, 128]
 *   v     (out)  [T, H, 128] f32 or bf16 (v_dtype): v[t, h] = o[t, h] @ w_vc[h],
 *                f32 accumulation.  Must not overlap the inputs.
 *   status       device word (may be NULL); DCP_STATUS_TIMEOUT as above.
 * Every pointer must be 16-byte aligned.  T == 0 is a no-op.  Errors:
 * DCP_ERR_INVALID as for dcp_absorb_q, or a bad dtype.
 */
int32_t dcp_absorb_o(int64_t T, int32_t H, const void* o, int32_t o_dtype, const void* w_vc, void* v,
                     int32_t v_dtype, int32_t* status, void* stream);

/*
 * dcp_lse_merge_absorb_o — the LSE merge and the output-side absorption
 * product in one call: v[t, h] = bf16(merged o[t, h]) @ w_vc[h].
 *
 * Sources: as dcp_lse_merge (the merge) and dcp_absorb_o (identity 2); "MLA 的
 * Decode Context Parallelism", section 4, stage 7 (the head owner merges the
 * partials and applies the V up-projection w_vc).  The merged latent output is
 * formed in shared memory as the tensor core's operand and never written out.
 *
 *   o_part    [n_parts, T, H, 512] f32 or bf16 (o_part_dtype): the partials,
 *             e.g. dcp_mla_decode_partial's o_part with T = B * q_len
 *   lse_part  f32 [n_parts, T, H] in base e (lse_base 0) or base 2 (1)
 *   w_vc      bf16 [H, 512, 128]
 *   v   (out) [T, H, 128] f32 or bf16 (v_dtype): f32 accumulation of the merged
 *             o, rounded to nearest bf16, times w_vc[h]
 *   lse (out) f32 [T, H], the merged lse in the partials' base (may be NULL)
 *   status    device word (may be NULL); DCP_STATUS_TIMEOUT if a pipeline wait
 *             gave up (v is then invalid)
 * A row whose parts are all empty gives v = 0 and lse = -inf.  T == 0 is a
 * no-op.  Errors: DCP_ERR_INVALID on n_parts outside [1, 64], T < 0, H outside
 * [1, 65535], a bad dtype or base, or a null / misaligned (16-byte) pointer.
 */
int32_t dcp_lse_merge_absorb_o(int32_t n_parts, int64_t T, int32_t H, const void* o_part, int32_t o_part_dtype,
                               const float* lse_part, int32_t lse_base, const void* w_vc, void* v, int32_t v_dtype,
                               float* lse, int32_t* status, void* stream);

/*
 * Exchange of the partials across W ranks (one GPU each).
 *
 * Sources: "Decode Context Parallelism" (zdszero), section "通信策略"
 * ("合并：All-to-All": each rank cuts O_r by head into one piece per rank and
 * sends it, with the matching LSE in the same buffer, to the rank that owns
 * those heads, which merges locally; "合并：AllGather + ReduceScatter": gather
 * every rank's LSE, correct each partial to exp(L_r - L) O_r, reduce-scatter the
 * corrected partials by head); "MLA 的 Decode Context Parallelism", section 4,
 * stages 6-7 and section 5 (the all-to-all carries bf16 o and an fp32 lse per
 * row, about 6.3 MB per rank and step at B=64, H=96).
 *
 * Rank w of W holds shards [w * n_held, (w + 1) * n_held) (n_held = N / W) and
 * owns heads [w * Hd, (w + 1) * Hd), Hd = H / W (H % W == 0).  Its partials are
 * dcp_mla_decode_partial's outputs for its shards: o_part [n_held, T, H, 512]
 * and lse_part [n_held, T, H], T = B * q_len query tokens.
 *
 * Wire format of the all-to-all: a send (or receive) buffer is [W][chunk],
 * chunk = dcp_a2a_chunk_bytes(...) bytes; chunk d of a send buffer holds an o
 * block [n_held, T, Hd, 512] in wire_dtype (bf16 rounded to nearest even, or
 * f32) for heads [d * Hd, (d + 1) * Hd), then an lse block [n_held, T, Hd] f32
 * right after the o block, padded to a multiple of 256 bytes.  After an
 * all-to-all with equal chunks (chunk w of the receive buffer came from rank w)
 * the receive buffer holds the head owner's rows of every shard in shard order.
 */

/* Bytes of one chunk (0 on bad arguments: n_held < 1, T < 0, H < 1, W < 1,
 * H % W != 0, a bad dtype). */
size_t dcp_a2a_chunk_bytes(int32_t n_held, int32_t T, int32_t H, int32_t world, int32_t wire_dtype);

/*
 * dcp_pack_partials — the send side of the all-to-all: chunk d of `send` gets
 * head slice d of every held shard's o_part (converted to wire_dtype) and
 * lse_part, in the wire format above.  o_part f32 or bf16 (o_part_dtype),
 * 16-byte aligned; send [world * chunk] bytes, 16-byte aligned (256 keeps every
 * chunk aligned).  Pad bytes are not written.  T == 0 is a no-op.  Errors:
 * DCP_ERR_INVALID as for dcp_a2a_chunk_bytes, or a null / misaligned pointer.
 */
int32_t dcp_pack_partials(int32_t n_held, int32_t T, int32_t H, int32_t world, const void* o_part,
                          int32_t o_part_dtype, const float* lse_part, void* send, int32_t wire_dtype,
                          void* stream);

/*
 * dcp_lse_merge_packed — the receive side: the exact LSE merge (as
 * dcp_lse_merge) of the world * n_held parts of each of `rows` = T * Hd rows,
 * read in place from an all-to-all receive buffer `recv` [world * chunk] in the
 * wire format (chunk w from rank w; part order = shard order).  o [rows, 512]
 * f32 or bf16 (o_dtype), i.e. [T, Hd, 512] of this rank's heads; lse f32 [rows]
 * in the partials' base (may be NULL).  rows == 0 is a no-op.  Errors:
 * DCP_ERR_INVALID on bad sizes, dtypes or base, or a null / misaligned pointer.
 */
int32_t dcp_lse_merge_packed(int32_t world, int32_t n_held, int64_t rows, const void* recv, int32_t wire_dtype,
                             int32_t lse_base, void* o, int32_t o_dtype, float* lse, void* stream);

/*
 * dcp_lse_rescale — the local step of the AllGather + ReduceScatter form.
 *
 *   lse_all   f32 [n_shards, T, H]: every shard's lse, shard order (the
 *             all-gather of each rank's lse_part)
 *   o_part    this rank's partials [n_held, T, H, 512], f32 or bf16
 *   o_sum     (out) f32 [world, T, Hd, 512]: block d, row (t, h') holds
 *             sum_{s held} base^(lse_{shard_begin+s} - L) * o_part[s, t, d*Hd + h']
 *             with L = log sum_r base^lse_r over all n_shards (the row's merged
 *             lse); a reduce-scatter (sum) of o_sum over the ranks leaves rank d
 *             the merged o of its heads
 *   lse       (out, may be NULL) f32 [world, T, Hd]: L in the same layout
 * A row whose shards are all empty gets o_sum = 0 and L = -inf.  T == 0 is a
 * no-op.  Errors: DCP_ERR_INVALID on bad sizes (shard_begin + n_held >
 * n_shards, H % world != 0, ...), dtype or base, or a null / misaligned pointer.
 */
int32_t dcp_lse_rescale(int32_t n_shards, int32_t shard_begin, int32_t n_held, int32_t T, int32_t H, int32_t world,
                        const float* lse_all, const void* o_part, int32_t o_part_dtype, int32_t lse_base,
                        float* o_sum, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DCP_H_ */
