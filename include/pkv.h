/*
 * pkv.h -- C ABI of libpkv: the paged-KV decode step of a Qwen3-style
 * attention layer on one GB300 (sm_103a).
 *
 * What the library computes is the attention half of the Qwen3-8B Nest
 * package's paged entries (qwen3-8b Nest files, src/attention.linnet,
 * GroupedQueryAttention.decode_paged and .step_paged; README.md, Entries):
 * for every token it
 *   1. applies per-head QK-norm, RMS normalisation of each head's head_dim
 *      slice with eps 1e-6 and a [head_dim] weight, to q and k (not v)
 *      (README.md; src/norm.linnet RmsNorm);
 *   2. rotates the normed q and k with rotate-half RoPE, base 1e6
 *      (src/rope.linnet tables; decode_paged's rope_rows);
 *   3. writes k and v at the token's slot of the page pool,
 *      slot = table[row][pos / page_size] * page_size + pos % page_size
 *      (decode_paged's page_slots + write_tokens);
 *   4. attends: query head h reads kv head h / (heads / kv_heads) over the
 *      row's positions 0..pos inclusive, scale 1/sqrt(head_dim)
 *      (decode_paged's paged_attention; decode_rows' mask s <= positions[b]).
 * The attention entries take the projected q, k, v split into heads
 * (split_heads: [tokens][heads][head_dim]) and return the attention output in
 * the same layout (merge_heads of it is a reshape).  The projections around
 * them are separate entries (pkv_qkv_proj before, pkv_linear for o_proj).
 *
 * Conventions shared by every entry point.
 *   - bf16 tensors are passed as void pointers to IEEE bfloat16 data.
 *   - "device" pointers must point into memory of the current CUDA device;
 *     "host" pointers into ordinary host memory.  The caller owns every
 *     tensor it passes; the library never frees them.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  pkv_decode,
 *     pkv_step and pkv_prefill only enqueue work on it: they neither allocate
 *     nor synchronise, and return before the GPU has run.
 *   - Errors a host check can see (null pointers, sizes, a workspace that is
 *     too small, an unsupported configuration) are returned synchronously as
 *     negative PKV_E* codes and nothing is enqueued.  Errors that depend on
 *     device-resident data (positions, page ids, slots) are caught on the
 *     device: the token is skipped (no write, zero output) and a bit is set
 *     in the pool's sticky error word, read with pkv_check_errors().  No
 *     kernel traps or spins without bound.
 *   - Optional host pre-check: with the environment variable PKV_CHECK=1,
 *     pkv_decode, pkv_decode_static, pkv_step and pkv_prefill first
 *     synchronise the stream, copy the call's positions, rows, slots and table
 *     to the host and return PKV_EINVAL (nothing enqueued) when two written
 *     slots coincide outside pool page 0, when a given prompt slot differs from
 *     table[rows[p]][positions[p] / page_size] * page_size + positions[p] % page_size,
 *     or, for the decode entries, when a row reads (at a position up to its
 *     own) a slot that another row of the call writes -- the one ordering
 *     decode does not provide (see pkv_decode).  Tokens the device checks
 *     would skip take no part.  The check is for debugging: it synchronises,
 *     so it does not belong in a captured graph.
 *   - Calls on one pool may run concurrently on different streams as long as
 *     they write different slots.  Each pkv_decode / pkv_step call takes one
 *     of the pool's 32 work counters in turn (zero between calls), so at most
 *     32 such calls may be in flight at once.
 *   - Every `table` argument may be NULL: the contiguous-row layout of the
 *     pages' non-paged entries (src/attention.linnet decode_rows,
 *     prefill_packed, step_packed), where row b owns the `pages` pool pages
 *     b * pages .. b * pages + pages - 1, so its position s sits at slot
 *     b * pages * page_size + s.  It needs rows * pages <= num_pages
 *     (PKV_ERANGE otherwise) and is otherwise the same as passing that
 *     identity table.
 *   - The kernels are built for head_dim 128, page_size 64 and
 *     heads == 4 * kv_heads (Qwen3-8B: 32 query heads over 8 kv heads); other
 *     shapes are rejected with PKV_ENOTIMPL at pool creation.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------------- */
#define PKV_OK 0
#define PKV_EINVAL (-1)     /* null pointer, non-positive size, misaligned buffer, bad config */
#define PKV_ERANGE (-2)     /* a size beyond what the library supports */
#define PKV_ENOMEM (-3)     /* device allocation failed (pool creation only) */
#define PKV_ECUDA (-4)      /* a CUDA runtime call failed */
#define PKV_EWORKSPACE (-5) /* workspace smaller than pkv_workspace_bytes() */
#define PKV_EDEVICE (-6)    /* no usable device, or the pool lives on another device */
#define PKV_ENOTIMPL (-7)   /* configuration the kernels are not built for */

/* ---- bits of the sticky device error word (pkv_check_errors) ---------------- */
#define PKV_DEVERR_POSITION 1u /* position < 0 (other than a -1 "no step"), >= max_seq, or >= pages*page_size */
#define PKV_DEVERR_PAGE 2u     /* a table entry the token reads is not in [0, num_pages) */
#define PKV_DEVERR_ROW 4u      /* a prompt token's row is not in [0, rows) */
#define PKV_DEVERR_SLOT 8u     /* an explicit prompt slot is not in [0, num_pages*page_size) */
#define PKV_DEVERR_TIMEOUT 16u /* a bounded device wait gave up (results of that call are void) */

/* ---- configuration ----------------------------------------------------------
 * Shape of one attention layer.  Defaults (pkv_config_default) are Qwen3-8B's:
 * qwen3-8b Nest files, nest.toml [generics] (Heads 32, KvHeads 8, HeadDim 128,
 * MaxSeq 40960), src/attention.linnet (PageSize 64), src/rope.linnet (THETA
 * 1e6), src/norm.linnet (eps 1e-6). */
typedef struct {
    int heads;         /* query heads per token */
    int kv_heads;      /* key/value heads per token */
    int head_dim;      /* elements per head vector */
    int page_size;     /* positions per page */
    int max_seq;       /* positions must be < max_seq (length of the RoPE table) */
    double rope_theta; /* RoPE base */
    double eps;        /* QK-norm epsilon */
    int rotary_dim;    /* RoPE rotates the first rotary_dim dims of each head (0 = all, the Qwen3 case);
                          the partial form of the gated-attention variant (fantasma model.zig, applyRope:
                          pairs (i, i + rotary_dim/2), inv_freq = theta^(-2i/rotary_dim)); built for
                          multiples of 32, PKV_ENOTIMPL otherwise */
} pkv_config;

/* Fill *cfg with the Qwen3-8B defaults.  Returns PKV_OK or PKV_EINVAL (null). */
PKV_API int pkv_config_default(pkv_config* cfg);

/* Human-readable name of a return code (static string, never NULL). */
PKV_API const char* pkv_strerror(int code);

/* ---- the page pool ------------------------------------------------------------
 * The pool is the layer's KV cache: with Batch 1 the cache's one row is a pool
 * of pages, page_size positions each, that rows reference through a page
 * table (README.md, Entries, decode_paged; src/lib.linnet Model.decode_paged).
 *
 * Layout of K and V (each): bf16 [kv_heads][num_pages * page_size][head_dim],
 * row-major.  Position s of page p for kv head g is element
 * ((g * num_pages + p) * page_size + s) * head_dim.  For one kv head a page is
 * one contiguous block of page_size * head_dim * 2 bytes (16 KiB).
 *
 * A pool also holds the RoPE (cos, sin) tables for positions 0..max_seq-1
 * (computed on the host in double precision and kept as fp32 hi + lo parts;
 * 16 bytes x head_dim/2 x max_seq, 42 MB at the defaults) and the sticky
 * device error word. */
typedef struct pkv_pool pkv_pool;

/* Create a pool that owns num_pages pages of K and V on the current device
 * (contents zeroed).  stream orders the initialisation.  *out receives the
 * pool; free it with pkv_pool_free.
 * Errors: PKV_EINVAL (null cfg/out, num_pages <= 0, bad config values),
 * PKV_ENOTIMPL (shape other than head_dim 128 / page_size 64 /
 * heads == 4*kv_heads), PKV_ERANGE (num_pages*page_size >= 2^31 or max_seq >
 * 2^20), PKV_ENOMEM, PKV_EDEVICE, PKV_ECUDA. */
PKV_API int pkv_pool_alloc(const pkv_config* cfg, int num_pages, void* stream, pkv_pool** out);

/* Create a pool over caller-owned K and V buffers (device pointers, layout as
 * above, 256-byte aligned).  The pool borrows them: the caller keeps them
 * alive until pkv_pool_free and frees them itself.  Their contents are left
 * as they are.  Errors as pkv_pool_alloc, plus PKV_EINVAL for a null or
 * misaligned k/v. */
PKV_API int pkv_pool_wrap(const pkv_config* cfg, int num_pages, void* k, void* v, void* stream, pkv_pool** out);

/* Release the pool (and its K/V if it owns them).  Waits for the device to
 * finish using it.  NULL is accepted and ignored. */
PKV_API int pkv_pool_free(pkv_pool* pool);

/* The pool's K and V device pointers and its number of slots
 * (num_pages * page_size).  Any output pointer may be NULL. */
PKV_API int pkv_pool_kv(const pkv_pool* pool, void** k, void** v, int64_t* num_slots);

/* ---- workspace ------------------------------------------------------------------
 * Scratch device memory a call needs, in bytes, for `tokens = prefill_tokens +
 * rows` tokens and a page table `pages` wide.  The caller allocates it (256-byte
 * aligned) and passes it to pkv_decode / pkv_step / pkv_prefill; its contents need no
 * initialisation and are not meaningful after the call.  The size depends
 * only on the pool (its config and attention grid size, see pkv_set_ctas),
 * rows and prefill_tokens: about 16.5 KiB per token plus 35 KiB per attention
 * CTA (room for the partial results of the pieces the work split makes), and
 * per prompt token heads * head_dim * 2 bytes more (8 KiB at the defaults) for
 * its queries, prepared once before the prompt attention.
 * Errors: PKV_EINVAL (null, rows < 0, prefill_tokens < 0, both zero,
 * pages <= 0), PKV_ERANGE (more than 2^20 tokens). */
PKV_API int pkv_workspace_bytes(const pkv_pool* pool, int rows, int pages, int prefill_tokens, size_t* bytes);

/* ---- decode_paged ------------------------------------------------------------------
 * qwen3-8b Nest files, src/attention.linnet GroupedQueryAttention.decode_paged
 * (steps 1-4 above) for `rows` rows, one new token each.  Row b's token sits
 * at position positions[b]; its key and value are written to
 *   slot = table[b][positions[b] / page_size] * page_size + positions[b] % page_size
 * and its query attends over positions 0..positions[b] of the row, read
 * through table[b] (so it sees its own new key).  All writes of the call
 * happen before any attention.
 *
 *   q         device bf16 [rows][heads][head_dim]     (projected, split into heads;
 *             16-byte aligned: its head groups are bulk-copied)
 *   k, v      device bf16 [rows][kv_heads][head_dim]
 *   q_norm_w  device bf16 [head_dim]                  (QK-norm weights)
 *   k_norm_w  device bf16 [head_dim]
 *   positions device int32 [rows]; -1 = the row takes no step (no write,
 *             zero output, not an error) -- the pages' own convention, a row
 *             that lists a scratch page, works as well
 *   table     device int32 [rows][pages], row-major; entries past a row's
 *             last page are never read.  NULL: contiguous rows (decode_rows)
 *   out       device bf16 [rows][heads][head_dim]
 *   workspace device, >= pkv_workspace_bytes(pool, rows, pages, 0), 256-byte aligned
 *
 * Slots written by one call must be distinct (the pages' write_tokens is a
 * scatter); if two tokens write one slot, which value lands is unspecified.
 * A row's new slot must not be read by another row of the same call (rows
 * may share pages, but only pages before their own write page, as a
 * shared prompt prefix is): each row's write is ordered before its own read,
 * not before other rows' reads.  pkv_step has no such condition.
 * Returns PKV_OK once the work is enqueued, or a PKV_E* code with nothing
 * enqueued. */
PKV_API int pkv_decode(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
               const void* k_norm_w, const int32_t* positions, const int32_t* table, int rows, int pages,
               void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ---- step_paged ----------------------------------------------------------------------
 * qwen3-8b Nest files, src/attention.linnet GroupedQueryAttention.step_paged:
 * P prompt tokens packed end to end (prefill_paged) and one step for each of
 * `rows` rows (decode_paged) in one pass.  Token order is the P prompt tokens,
 * then the rows' step tokens.  Prompt token p sits at position positions[p]
 * of table row prow[p] and is written at slots[p]; row b's step token sits at
 * step_positions[b].  All P + rows tokens are normed, roped and written
 * first; then prompt token p attends over table[prow[p]] for positions
 * 0..positions[p] (its own chunk's earlier keys included), and row b over
 * 0..step_positions[b].
 *
 *   q              device bf16 [P + rows][heads][head_dim], 16-byte aligned
 *   k, v           device bf16 [P + rows][kv_heads][head_dim]
 *   positions      device int32 [P]
 *   prow           device int32 [P]    (the pages' `rows` argument)
 *   slots          device int32 [P], or NULL: derive each slot from the table
 *   step_positions device int32 [rows]; -1 = row takes no step
 *   table          device int32 [rows][pages], or NULL: contiguous rows (step_packed)
 *   out            device bf16 [P + rows][heads][head_dim] (prompts, then steps), 16-byte aligned
 *   workspace      >= pkv_workspace_bytes(pool, rows, pages, P)
 * The pages require P > 0 and rows > 0 (PKV_EINVAL otherwise).  Slots must
 * be distinct as for pkv_decode; every write of the call is ordered before
 * every read. */
PKV_API int pkv_step(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
             const void* k_norm_w, const int32_t* positions, const int32_t* prow, const int32_t* slots,
             const int32_t* step_positions, const int32_t* table, int P, int rows, int pages, void* out,
             void* workspace, size_t workspace_bytes, void* stream);

/* ---- prefill_paged -------------------------------------------------------------------
 * qwen3-8b Nest files, src/attention.linnet GroupedQueryAttention.prefill_paged:
 * P prompt tokens packed end to end, no step tokens.  Prompt token p sits at
 * position positions[p] of table row prow[p] and is written at slots[p]; all
 * P tokens are normed, roped and written first, then token p attends over
 * table[prow[p]] for positions 0..positions[p].  A prompt may continue a row
 * (a later chunk of a long prompt, or a prompt after a shared prefix whose
 * pages the row lists): it sees every key the row already holds below its
 * position as well as its own chunk's.
 *
 *   q          device bf16 [P][heads][head_dim], 16-byte aligned
 *   k, v       device bf16 [P][kv_heads][head_dim]
 *   positions  device int32 [P]
 *   prow       device int32 [P]    (the pages' `rows` argument)
 *   slots      device int32 [P], or NULL: derive each slot from the table
 *   table      device int32 [rows][pages], or NULL: contiguous rows.  With a
 *              NULL table and every prompt filling its own row from position 0,
 *              this is prefill_packed with segments = prow.
 *   out        device bf16 [P][heads][head_dim], 16-byte aligned
 *   workspace  >= pkv_workspace_bytes(pool, 0, pages, P)
 * P > 0 and rows > 0 (PKV_EINVAL otherwise); `rows` bounds prow[p].  Slots must
 * be distinct; every write of the call is ordered before every read. */
PKV_API int pkv_prefill(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
                        const void* k_norm_w, const int32_t* positions, const int32_t* prow, const int32_t* slots,
                        const int32_t* table, int P, int rows, int pages, void* out, void* workspace,
                        size_t workspace_bytes, void* stream);

/* ---- the projections either side: linear layers -------------------------------------
 * qwen3-8b Nest files, src/attention.linnet GroupedQueryAttention.decode_paged and
 * step_paged: q_proj, k_proj and v_proj map the layer input x [tokens][hidden] to
 * q [tokens][heads * head_dim] and k, v [tokens][kv_heads * head_dim] (split_heads
 * of these is the [tokens][heads][head_dim] layout pkv_decode / pkv_step take, a
 * reshape), and o_proj maps merge_heads of their output back to [tokens][hidden].
 * None has a bias (README.md).  One call computes one of them:
 *   y[t][o] = sum_k x[t][k] * w[o][k]   (bf16 inputs, fp32 accumulation, bf16 output)
 *
 *   x          device bf16 [tokens][in_features], in_features % 64 == 0, 16-byte aligned
 *   w          device bf16 [out_features][in_features] (nn.Linear layout), out_features % 128 == 0
 *   y          device bf16 [tokens][out_features], 16-byte aligned
 *   workspace  device, >= pkv_linear_workspace_bytes(...), 256-byte aligned: 0 bytes in
 *              this version (may be NULL): when few tokens leave SMs idle, the input
 *              features are split over the CTAs of a cluster, which sum their fp32
 *              partial tiles in shared memory
 * The pool names the device and receives device errors; nothing of it is read.
 * Other feature counts return PKV_ENOTIMPL; returns once the work is enqueued. */
PKV_API int pkv_linear_workspace_bytes(const pkv_pool* pool, int tokens, int in_features, int out_features,
                                       size_t* bytes);
PKV_API int pkv_linear(pkv_pool* pool, const void* x, const void* w, void* y, int tokens, int in_features,
                       int out_features, void* workspace, size_t workspace_bytes, void* stream);

/* The three projections before the attention in one launch: w_qkv is q_proj,
 * k_proj and v_proj stacked row-wise, [(heads + 2 kv_heads) * head_dim][hidden]
 * (the pool's config), and
 *   q[t] = x[t] Wq^T  [tokens][heads][head_dim]
 *   k[t] = x[t] Wk^T  [tokens][kv_heads][head_dim]
 *   v[t] = x[t] Wv^T  [tokens][kv_heads][head_dim]
 * the layouts pkv_decode / pkv_step / pkv_prefill take.  Same arithmetic as
 * pkv_linear; hidden % 64 == 0 (PKV_ENOTIMPL otherwise); all pointers 16-byte
 * aligned device memory. */
PKV_API int pkv_qkv_proj(pkv_pool* pool, const void* x, const void* w_qkv, int tokens, int hidden, void* q, void* k,
                         void* v, void* stream);

/* ---- the projection with the per-token work fused in, and the attention after it --------
 * qwen3-8b Nest files, src/attention.linnet, GroupedQueryAttention.decode_paged:
 *   q = rope_rows(q_norm(split_heads(q_proj(x))))
 *   k = rope_rows(k_norm(split_heads(k_proj(x)))),  v = split_heads(v_proj(x))
 *   write_tokens(k, v at page_slots(table, positions))
 * in one launch, for `tokens` decode rows (token t is table row t, at
 * positions[t]): the product of pkv_qkv_proj, whose epilogue -- each 128-feature
 * tile of the product is one head, all of it in the CTA that finishes it --
 * rounds q, k, v to bf16 (the pages' projection outputs), applies QK-norm and
 * RoPE to q and k exactly as pkv_decode does, writes k and v to their slots of
 * the pool and q to q_hat.  The raw q, k, v never reach memory.
 *   x, w_qkv   as pkv_qkv_proj (hidden % 64 == 0, PKV_ENOTIMPL otherwise)
 *   q_norm_w, k_norm_w  device bf16 [head_dim]
 *   positions  device int32 [tokens]; -1 = no step (nothing written)
 *   table      device int32 [tokens][pages], or NULL (contiguous rows)
 *   q_hat      device fp32 [tokens][heads][head_dim], 16-byte aligned (out):
 *              QK-normed, roped q, unscaled
 * Rows whose position or pages pkv_decode would reject are not written and set
 * the same device error bits.  Slots must be distinct (PKV_CHECK=1 checks).
 * Follow it with pkv_decode_appended on the same stream. */
PKV_API int pkv_qkv_proj_append(pkv_pool* pool, const void* x, const void* w_qkv, int tokens, int hidden,
                                const void* q_norm_w, const void* k_norm_w, const int32_t* positions,
                                const int32_t* table, int pages, float* q_hat, void* stream);

/* decode_paged's attention for rows whose q was prepared and whose k and v
 * were appended by pkv_qkv_proj_append (the same positions and table): row b
 * attends over positions 0..positions[b] of table[b], with q_hat[b] (fp32
 * [rows][heads][head_dim]).  Nothing is written to the pool, so rows may
 * read each other's new slots (the call that wrote them has completed before
 * this one on the stream).  Workspace, output, skipped rows and error bits as
 * pkv_decode. */
PKV_API int pkv_decode_appended(pkv_pool* pool, const float* q_hat, const int32_t* positions, const int32_t* table,
                                int rows, int pages, void* out, void* workspace, size_t workspace_bytes,
                                void* stream);

/* ---- output gate of the gated-attention variant ----------------------------------------
 * fantasma model.zig, fullAttentionForward ("Full Attention (GQA with output gate +
 * QK-norm + partial RoPE)"): the q projection also yields a gate per head and
 * dim, and the attention output is multiplied by its sigmoid before o_proj:
 *   out[t][h][d] *= 1 / (1 + exp(-gate[t][h][d]))     (fp32, rounded to bf16)
 * With a pool whose rotary_dim is below head_dim (the variant's partial RoPE),
 * pkv_decode / pkv_step / pkv_prefill followed by this call give that layer's
 * attention.  Qwen3-8B has no gate.
 *   out   device bf16 [tokens][heads][head_dim], updated in place, 16-byte aligned
 *   gate  device bf16 [tokens][heads][head_dim], 16-byte aligned */
PKV_API int pkv_output_gate(pkv_pool* pool, void* out, const void* gate, int tokens, void* stream);

/* ---- decode without a caller workspace -------------------------------------------------------
 * The pages have no counterpart to this entry point; it is a convenience of
 * this library.  It is pkv_decode for callers that cannot allocate device
 * memory at all: for example a plug-in whose host application owns every
 * device allocation and hands it none, or a process whose device memory is
 * reserved in full up front by another allocator, where one more cudaMalloc
 * would fail, or would stall the whole device while it runs.
 *
 * Instead of a caller workspace it uses a scratch array compiled into the
 * library: PKV_STATIC_SCRATCH_BYTES (32 MiB) of device memory that every GPU
 * that loads the library holds until the process exits.  The call itself
 * allocates no device memory.  The caller still passes the pool, inputs and
 * output, exactly as for pkv_decode (same layouts, same error codes, the same
 * PKV_CHECK=1 debugging pre-check, which copies the call's tables into host
 * memory), minus the workspace.
 *   - Each call whose stream is not being captured looks up the array's
 *     device address on the current device (so the array reloaded after a
 *     cudaDeviceReset is found again); a call under stream capture reuses the
 *     address the last uncaptured call on that device found.  Make one call
 *     on each device before capturing any.
 *   - Every call shares the one array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero.  Calls whose work overlaps on the
 *     GPU (e.g. on two streams with no ordering between them) race on the array
 *     and their results are undefined.
 *   - A call that needs more scratch than the array holds (more than
 *     PKV_STATIC_SCRATCH_BYTES from pkv_workspace_bytes(pool, rows, pages, 0))
 *     is rejected with PKV_ERANGE and nothing is enqueued. */
#define PKV_STATIC_SCRATCH_BYTES (32u << 20)
PKV_API int pkv_decode_static(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
                              const void* k_norm_w, const int32_t* positions, const int32_t* table, int rows,
                              int pages, void* out, void* stream);

/* ---- errors ------------------------------------------------------------------------------
 * Synchronise `stream`, then read and clear the pool's sticky device error
 * word (PKV_DEVERR_* bits of every call since the last read) into *flags.
 * Returns PKV_ECUDA if the stream reports a CUDA error. */
PKV_API int pkv_check_errors(pkv_pool* pool, void* stream, uint32_t* flags);

/* ---- tuning and measurement ---------------------------------------------------------------
 * Grid size of the attention kernel (0 = one wave: every SM's resident
 * CTAs).  The kernel cuts the call's (token, kv head, page) sequence into
 * that many equal slices of about three quarters of it, one per CTA, and
 * chunks of 4+ pages of the rest that the CTAs claim as they finish (with one
 * CTA, a single slice).  Results are reproducible run to run and do not
 * depend on the grid size beyond floating-point association.  It changes
 * pkv_workspace_bytes.  Errors: PKV_EINVAL (null, < 0). */
PKV_API int pkv_set_ctas(pkv_pool* pool, int ctas);

/* Limit, in nanoseconds, of each bounded wait inside the decode attention
 * kernel (the shared-memory ring between its copy warp and its compute warps,
 * and the compute warps' meeting points); default 1e9 (one second).  A wait
 * that runs out makes its CTA stop: it sets PKV_DEVERR_TIMEOUT in the error
 * word, lets the copies it has in flight land (allowing a full second for
 * that, whatever this limit), and exits; the outputs of that call are void,
 * and the pool is ready for the next call.  0 gives up at the first check
 * that finds the awaited data not yet there, which lets a test run the
 * timeout path on purpose.  Applies to calls enqueued after it.
 * Errors: PKV_EINVAL (null, ns < 0). */
PKV_API int pkv_set_wait_limit(pkv_pool* pool, int64_t ns);

/* Kernel timer: while enabled, every pkv_decode / pkv_step records a pair of
 * CUDA events on its stream around the decode attention kernel (the dominant
 * launch), every pkv_prefill around its prompt-attention kernel and every
 * pkv_linear around its matrix-product kernel.  pkv_timer_read synchronises on the last recorded event,
 * returns the summed duration in milliseconds and the number of timed
 * launches since the timer was last enabled, and keeps the timer running.
 * At most 4096 launches are kept (later ones overwrite the oldest).
 * enable: 0 off, 1 every launch named above, 2 the attention launches only
 * (not pkv_linear / pkv_qkv_proj / pkv_qkv_proj_append); PKV_EINVAL otherwise.  Host
 * threads sharing a pool take distinct event slots; pkv_timer_enable and
 * pkv_timer_read should not race with calls in flight on other threads.
 * A timed pkv_step runs its prompt attention and its step rows' attention one
 * after the other (the events between them), where an untimed one runs them
 * side by side on a split of the SMs: the timer measures the rows' attention
 * alone, not the step. */
PKV_API int pkv_timer_enable(pkv_pool* pool, int enable);
PKV_API int pkv_timer_read(pkv_pool* pool, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
