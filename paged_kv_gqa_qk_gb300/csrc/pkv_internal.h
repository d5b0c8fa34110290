// Internal declarations shared by the host API and the kernel translation
// units of libpkv.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pkv.h"

namespace pkv {

// Shapes the kernels are built for (Qwen3-8B attention).
constexpr int kHeadDim = 128;
constexpr int kPageSize = 64;
constexpr int kGroup = 4;                                  // query heads per kv head
constexpr int kPageBytes = kPageSize * kHeadDim * 2;       // one page of K (or V) for one kv head
constexpr int kRopeHalf = kHeadDim / 2;
// The score scale the prompt attention's queries carry: log2(e) / sqrt(128), so that
// its scores are in base-2 units.
constexpr float kQScale = 1.4426950408889634f * 0.088388347648318440f;

constexpr int kTimerSlots = 4096;

// The attention kernel's work split (see split_of in the kernels): after its
// static slice a CTA claims chunks from a counter; at most kDynChunksPerCta
// chunks per CTA, kept in one of kClaimSlots counters that calls take in turn.
constexpr int kDynChunksPerCta = 16;
constexpr int kClaimSlots = 32;

}  // namespace pkv

struct pkv_pool {
    pkv_config cfg;
    int device;
    int num_sms;
    int num_pages;
    int64_t num_slots;
    bool owns_kv;
    void* k;               // bf16 [kv_heads][num_slots][head_dim]
    void* v;
    float2* rope_hi;       // (cos, sin) [max_seq][head_dim/2]: fp32 nearest to the double values
    float2* rope_lo;       // the double values minus rope_hi, in fp32
    uint32_t* err;         // sticky device error word (word 0 of a 256-byte allocation)
    uint32_t* claims;      // kClaimSlots chunk counters (bytes 128..255 of the same allocation), zero between calls
    std::atomic<uint64_t> call_seq;  // calls enqueued (from any host thread): call n uses claims[n % kClaimSlots]
    CUtensorMap tmap_k;    // 3-D tiled view of K: {head_dim, num_slots, kv_heads}, box {64, 64, 1}, 128B swizzle
    CUtensorMap tmap_v;
    int ctas_per_sm;       // resident attention CTAs per SM (occupancy)
    int ctas_override;     // attention grid size; 0 = one wave (ctas_per_sm x SMs)
    uint64_t wait_ns;      // limit of the decode attention kernel's ring and group waits (default 1 s)
    // kernel timer: a timed call takes event slot timer_count++ % kTimerSlots (atomic,
    // so host threads sharing the pool take distinct slots)
    int timer_on;          // 0 off, 1 every timed launch, 2 the attention launches only
    std::atomic<int64_t> timer_count;
    cudaEvent_t* ev_start;
    cudaEvent_t* ev_stop;
};

namespace pkv {

// Workspace carve-up for one call (all offsets 256-byte aligned).
struct Plan {
    int tokens;         // P + rows
    int pages;          // table width
    int ctas;           // attention grid size C
    size_t off_len, off_row, off_prefix, off_unit_ok, off_po, off_plse;
    size_t off_sched;   // prompt attention: counter of claimed work units (zeroed by prep_kernel)
    size_t off_qhat;    // prompt tokens' queries after QK-norm, RoPE and kQScale: bf16 [P][heads][128]
    uint32_t* claim;    // decode attention: this call's chunk counter (reset by combine_kernel)
    size_t total;
};

Plan make_plan(const pkv_pool* pool, int tokens, int pages, int prompt_tokens);

// Arguments of one decode/step call after host validation.
struct StepArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* q_norm_w;
    const void* k_norm_w;
    const int32_t* positions;       // [P]  (prompt tokens)
    const int32_t* prow;            // [P]
    const int32_t* slots;           // [P] or null
    const int32_t* step_positions;  // [steps]
    const int32_t* table;           // [rows][pages], or null: row b owns pages b*pages .. b*pages + pages - 1
    int P;                          // prompt tokens
    int rows;                       // table rows
    int pages;                      // table width
    int steps;                      // step tokens (rows for decode and step, 0 for prefill)
    void* out;
    char* ws;
    const float* q_hat;             // decode with q prepared and k/v appended beforehand, or null
};

// An NVTX range over one entry-point call (its host-side enqueue), for
// timeline tools; a no-op unless a tool is attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Pool page holding page j of table row `row` (a null table: contiguous rows).
__device__ __forceinline__ int page_of(const int32_t* table, int pages, int row, int j)
{
    return table ? table[(int64_t)row * pages + j] : row * pages + j;
}

// A step's SMs, split between the prompt attention and the step rows' attention.
// The prompt attention keeps prompt_sms(...) SMs and the rows' attention starts
// on the others at once (it is launched when every prompt-attention CTA has
// started, so its CTAs land on the SMs the ones beyond the kept count leave);
// both kernels derive the split from the same token lengths, so they agree.
// Costs are in 1/25 µs of one SM: a prompt unit (64-token tile, kv head) 6.4 µs
// plus 1.12 µs a page of its longest token (the prompt attention's measured
// rate, start and tail included), a step row's page of one kv head 0.52 µs (32
// KiB at ~60 GB/s, what one SM streams when the rows have part of the chip).
constexpr int64_t kSplitPromptUnit = 160, kSplitPromptPage = 28, kSplitRowPage = 13;
constexpr int kSplitMinRowSms = 8;  // leaving the rows fewer SMs than this: no split

__host__ __device__ inline int prompt_sms(int64_t prompt_cost, int64_t row_cost, int prompt_units, int sms)
{
    if (prompt_cost <= 0 || row_cost <= 0) return sms;
    int n = (int)((prompt_cost * sms + (prompt_cost + row_cost) / 2) / (prompt_cost + row_cost));
    const int few = prompt_units < sms / 4 ? prompt_units : sms / 4;  // each of a few units its own SM
    n = n > few ? n : few;
    if (n < 1) n = 1;
    return n > sms - kSplitMinRowSms ? sms : n;
}

// Cost of one prompt tile (whose tokens' attended lengths have maximum max_len)
// in the units above, over its kv heads; 0 for a tile with no token.
__host__ __device__ inline int64_t prompt_tile_cost(int max_len, int kv_heads)
{
    return max_len > 0 ? (int64_t)kv_heads * (kSplitPromptUnit + kSplitPromptPage * ((max_len + kPageSize - 1) / kPageSize))
                       : 0;
}

// 2-D tiled tensor map of a row-major bf16 matrix (128-byte swizzle, zero fill
// past the edges); false if the driver refuses it.
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer);
// 3-D tiled tensor map {128 dims, heads, tokens} of bf16 [tokens][heads][128]; a box
// is 64 dims (the 128-byte swizzle span) x 1 head x 32 tokens, zero fill past the
// last token.
bool make_tmap_heads(CUtensorMap* map, const void* base, int heads, int tokens);

// y = x W^T (pkv_linear): tokens per tile, input-feature splits (CTAs of one
// cluster), and the launch.
int linear_tile_tokens(int tokens);
int linear_splits(const pkv_pool* pool, int tokens, int in, int out);
cudaError_t launch_linear(pkv_pool* pool, const void* x, const void* w, int tokens, int in, int nseg,
                          void* const* y, const int* widths, cudaStream_t s);

// pkv_qkv_proj_append: the q/k/v projection of `tokens` decode rows (token t =
// table row t) with QK-norm, RoPE and the k/v append done by its epilogue.
struct QkvAppend {
    const void* q_norm_w;
    const void* k_norm_w;
    const int32_t* positions;  // [tokens]
    const int32_t* table;      // [tokens][pages], or null (contiguous rows)
    int pages;
    float* q_hat;              // [tokens][heads][head_dim] fp32 out
};
cudaError_t launch_qkv_append(pkv_pool* pool, const void* x, const void* w_qkv, int tokens, int hidden,
                              const QkvAppend& a, cudaStream_t s);

// out *= sigmoid(gate) over n bf16 elements (n % 8 == 0, 16-byte aligned).
cudaError_t launch_gate(const pkv_pool* pool, void* out, const void* gate, int64_t n, cudaStream_t s);

// Per-device kernel attributes (dynamic shared memory); called with the
// pool's device current when a pool is created.
cudaError_t configure_kernels();
cudaError_t configure_prefill();
// Resident attention CTAs per SM (0 on error).
int attn_ctas_per_sm();

// Kernel launchers (pkv_kernels.cu).  Each returns a cudaError_t from the launch.
//   decode: attn (decode mode, fuses validation + append) -> combine
//   step:   prep (validation + append of every token) -> attn (step mode) -> combine
cudaError_t launch_prep(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s);
cudaError_t launch_attn(const pkv_pool* pool, const StepArgs& a, const Plan& plan, bool decode_mode, bool pdl,
                        cudaStream_t s);
cudaError_t launch_combine(const pkv_pool* pool, const StepArgs& a, const Plan& plan, bool decode_mode,
                           cudaStream_t s);
// step mode: prompt-token attention on tcgen05 tensor cores (pkv_prefill.cu), a
// persistent grid of `ctas` CTAs (one per SM; capped at its work units)
// split: the step rows' attention is launched beside it (programmatic launch); the
// kernel then keeps only prompt_sms(...) of its CTAs (see prompt_sms).
cudaError_t launch_prefill(const pkv_pool* pool, const StepArgs& a, const Plan& plan, int ctas, bool split,
                           cudaStream_t s);

// Enqueue one decode (a.P == 0) or step call on workspace a.ws; host checks done.
int enqueue(pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s);

// The optional host pre-check (environment variable PKV_CHECK=1): synchronises
// s, copies the call's token tables to the host and returns PKV_EINVAL for a
// call whose written slots coincide outside page 0, whose given prompt slots
// disagree with the table, or (decode) whose rows read another row's new slot.
bool check_enabled();
int host_precheck(const pkv_pool* pool, const StepArgs& a, cudaStream_t s);

}  // namespace pkv
