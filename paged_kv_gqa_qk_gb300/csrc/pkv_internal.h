// Internal declarations shared by the host API and the kernel translation
// units of libpkv.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// Shapes the kernels are built for (Qwen3-8B attention).
constexpr int kHeadDim = 128;
constexpr int kPageSize = 64;
constexpr int kGroup = 4;                                  // query heads per kv head
constexpr int kPageBytes = kPageSize * kHeadDim * 2;       // one page of K (or V) for one kv head
constexpr int kRopeHalf = kHeadDim / 2;

constexpr int kTimerSlots = 4096;

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
    double2* rope;         // (cos, sin) [max_seq][head_dim/2], double precision
    uint32_t* err;         // sticky device error word
    CUtensorMap tmap_k;    // 3-D tiled view of K: {head_dim, num_slots, kv_heads}, box {64, 64, 1}, 128B swizzle
    CUtensorMap tmap_v;
    int split_pages;       // 0 = automatic
    // kernel timer
    bool timer_on;
    int64_t timer_count;
    cudaEvent_t* ev_start;
    cudaEvent_t* ev_stop;
};

namespace pkv {

// Workspace carve-up for one call (all offsets 256-byte aligned).
struct Plan {
    int tokens;         // P + rows
    int pages;          // table width
    int chunk;          // pages per split
    int max_splits;     // ceil(pages / chunk)
    size_t off_len, off_row, off_qhat, off_po, off_plse, total;
};

Plan make_plan(const pkv_pool* pool, int tokens, int pages);

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
    const int32_t* step_positions;  // [rows]
    const int32_t* table;           // [rows][pages]
    int P;
    int rows;
    int pages;
    void* out;
    char* ws;
};

// Per-device kernel attributes (dynamic shared memory); called with the
// pool's device current when a pool is created.
cudaError_t configure_kernels();

// Kernel launchers (pkv_kernels.cu).  Each returns a cudaError_t from the launch.
cudaError_t launch_prep(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s);
cudaError_t launch_attn_decode(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s);
cudaError_t launch_combine(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s);

}  // namespace pkv
