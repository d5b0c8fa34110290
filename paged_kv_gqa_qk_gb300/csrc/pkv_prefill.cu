// Prompt-chunk attention of step_paged / prefill_paged on tcgen05 tensor
// cores (sm_103a).
//
// qwen3-8b Nest files, src/attention.linnet, GroupedQueryAttention.step_paged
// and prefill_paged: after every token of the call has been written to the
// pool (prep_kernel), prompt token p attends over table[rows[p]] for
// positions 0..positions[p] -- its own chunk's earlier keys included.
//
// Work unit: a tile of 64 consecutive prompt tokens and one kv head g.  The
// tile is two halves of 32 tokens, one per softmax group; in each half the 4
// query heads of g times the 32 tokens are the M = 128 rows of the products,
// row m = head (m / 32) of the group, token (m % 32) of the half, so
// tensor-memory lane m belongs to thread m of the group's four warps.  Both
// halves read the same blocks of two pages (128 keys) of the row; per block b:
//   S_h  = Q_h K_b^T         128 x 128, K = 128 dims   (tcgen05, into TMEM)
//   P_h  = 2^(S_h - m_h)     causal mask, online max   (softmax group h, bf16
//                            back into TMEM over the first half of S_h)
//   O_h += P_h V_b           128 x 128, K = 128 keys   (tcgen05, A from TMEM)
// Q carries the QK-norm, the RoPE and the score scale log2(e)/sqrt(128), so S
// is in base-2 units; prep_kernel prepares it once per token, and each unit
// copies its 64 tokens x 4 heads into shared memory with the tensor-copy
// engine (16 boxes of 32 tokens x 64 dims of one head, swizzled as the
// products read them).  The running max only moves (and O, l are rescaled in
// place) when a block raises it by more than 8: in between, P stays below 2^8.
//
// The two groups ping-pong: the tensor cores run one group's products while
// the other group's softmax runs.  The issuing order per block is
//   PV_0(b), S_0(b+1), PV_1(b), S_1(b+1)
// so that S_h(b+1), which overwrites P_h(b) in tensor memory, is issued after
// the product that reads it (tcgen05 operations of one thread run in order).
//
// Warp roles: 0-3 softmax group 0, 4-7 softmax group 1 (each also writes its
// outputs), 8 TMA producer (each unit's Q, then the K and the V of each block
// through a ring of four 32 KiB stages), 9 tensor-memory allocation and the
// MMA-issuing thread.
//
// The grid is persistent, one CTA per SM.  Units are taken from a counter in
// the workspace in decreasing order of the tile's page count (longest first),
// an order every CTA derives identically from the token table.  A tile whose
// tokens belong to several table rows (where one prompt ends and the next
// begins) is processed once per row; tokens of the other rows are masked out
// of that pass.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {

constexpr uint32_t kAll = 0xffffffffu;
constexpr int kHalfTok = 32;                   // tokens of one half (one softmax group)
constexpr int kTileTok = 2 * kHalfTok;         // tokens of a tile
constexpr int kRowsM = kHalfTok * kGroup;      // 128 = M of every product
constexpr int kBlockKeys = 2 * kPageSize;      // keys of a block: two pages
constexpr int kPfStages = 4;                   // ring stages, each the K or the V of one block
constexpr int kPfStageBytes = kBlockKeys * kHeadDim * 2;  // 32 KiB
constexpr int kHalfBytes = kPfStageBytes / 2;  // one 64-dim half of a stage: [2 pages][64 keys][128 B]
constexpr int kGroups = 2;
constexpr int kProducer = 4 * kGroups, kIssuer = kProducer + 1;
constexpr int kPfThreads = 32 * 4 * (kGroups + 1);  // three warpgroups; warps 10 and 11 only take part in barriers
// Registers per thread: the launch gives every thread kRegsLaunch; the third
// warpgroup (producer, issuer) hands registers to the two softmax groups.
constexpr uint32_t kRegsLaunch = 168, kRegsSoftmax = 200, kRegsOther = 104;
static_assert(kGroups * 128 * kRegsSoftmax + 128 * kRegsOther <= kPfThreads * kRegsLaunch, "register split");
static_assert(kRegsLaunch * kPfThreads <= 65536, "register file");
constexpr uint32_t kTmemCols = 512;            // group h: S/P at 256h, O at 256h + 128
constexpr float kRescale = 8.f;                // log2 headroom before the running max moves
constexpr int kMaxSortTiles = 2048;            // larger calls take tiles in token order
// sort key of a work item (tile, run): pages << 17 | (2047 - tile) << 6 | (63 - run)
constexpr int kKeyTileShift = 6, kKeyPagesShift = 17;

struct PfSmem {
    static constexpr int kQ = 0;                                    // 2 groups x [2 halves][128 rows][128 B]
    static constexpr int kRing = kQ + kGroups * 2 * kRowsM * 128;   // stages x 32 KiB
    static constexpr int kSort = kRing + kPfStages * kPfStageBytes;  // uint32 [kMaxSortTiles]
    static constexpr int kTok = kSort + 4 * kMaxSortTiles;          // int pos[64], row[64]
    static constexpr int kRuns = kTok + 2 * kTileTok * 4;           // int row[64], npages[64], count, unit
    static constexpr int kSplit = kRuns + (2 * kTileTok + 4) * 4;   // u64 prompt cost, prompt units, row pages
    static constexpr int kBars = kSplit + 32;
    // full[S], empty[S], s_ready[2], p_ready[2], o_done[2], epi[2], drain, q_full
    static constexpr int kNumBars = 2 * kPfStages + 4 * kGroups + 2;
    static constexpr int kTmemSlot = kBars + 8 * kNumBars;
    static constexpr int kFlag = kTmemSlot + 16;
    static constexpr int kBytes = kFlag + 16;
    static constexpr int kAlloc = kBytes + 1024;
};
static_assert(PfSmem::kAlloc <= 227 * 1024, "prefill shared memory");
constexpr int kQBytes = kGroups * 2 * kRowsM * 128;  // a unit's Q: 64 tokens x 4 heads x 128 dims, bf16

struct PfParams {
    const int32_t* tok_len;   // [P] attended length from prep_kernel, 0 = skip
    const int32_t* tok_row;   // [P]
    const int32_t* table;     // [rows][pages], or null (contiguous rows)
    __nv_bfloat16* out;       // [P + rows][heads][128]
    int32_t* sched;           // unit counter, zero at launch
    uint32_t* err;
    int P, pages, heads, kv_heads, ntiles;
    int split;                // 1: the step rows' attention runs beside this grid (see prompt_sms); the
                              // kernel instantiated with kSplit = true runs it
    int steps, sms;           // the step rows (tokens P..P+steps-1 of the token table), the device's SMs
};


// Shared-memory addresses and launch-wide values every role needs.
struct PfCtx {
    uint32_t base;   // 1024-aligned shared address of the layout
    uint8_t* sbase;  // the same, generic
    uint32_t bar_full, bar_empty, bar_s, bar_p, bar_o, bar_epi, bar_drain, bar_q;
    uint32_t tmem;
    int* sPos;
    int* sRow;
    int* sRunRow;
    int* sRunPages;
    int* sNumRuns;
    int* sUnit;
    const uint32_t* sKey;
    volatile int* abort_flag;
    int nunits;
    bool sorted;
};

// Work unit u: kv head u % G of item u / G; an item is one run (table row) of
// a tile when the items are sorted, else a whole tile (every run, run = -1).
__device__ __forceinline__ void item_of(const PfCtx& c, const PfParams& p, int u, int& tile, int& run)
{
    if (c.sorted) {
        const uint32_t key = c.sKey[u / p.kv_heads];
        tile = (kMaxSortTiles - 1) - (int)((key >> kKeyTileShift) & (kMaxSortTiles - 1));
        run = 63 - (int)(key & 63);
    } else {
        tile = u / p.kv_heads;
        run = -1;
    }
}

// The runs of a tile (one per table row among its valid tokens, in order of
// first token) computed by one warp; lane l holds tokens l and l + 32 with
// positions pa, pb and rows ra, rb (position < 0: not a token).  For each run
// calls emit(index, row, pages) on every lane; returns the number of runs.
template <typename Emit>
__device__ __forceinline__ int tile_runs(int pa, int pb, int ra, int rb, Emit emit)
{
    bool ua = pa >= 0, ub = pb >= 0;  // valid tokens not yet in a run
    int nr = 0;
    for (;;) {
        const uint32_t ma = __ballot_sync(kAll, ua), mb = __ballot_sync(kAll, ub);
        if (!ma && !mb) break;
        const int r = ma ? __shfl_sync(kAll, ra, __ffs(ma) - 1) : __shfl_sync(kAll, rb, __ffs(mb) - 1);
        const bool ia = ua && ra == r, ib = ub && rb == r;
        const int n = (int)__reduce_max_sync(
            kAll, (uint32_t)max(ia ? pa / kPageSize + 1 : 0, ib ? pb / kPageSize + 1 : 0));
        emit(nr, r, n);
        ua = ua && !ia;
        ub = ub && !ib;
        ++nr;
    }
    return nr;
}

// S_h = Q_h K^T for the block of npg pages in the ring stage at `kst`, into
// group h's S columns; its completion arrives on s_ready[h].  A descriptor of
// k-step k is the k = 0 one plus the step's byte offset / 16 (no carry: shared
// addresses stay below 2^18).
__device__ __forceinline__ void issue_s(uint32_t tmem, uint32_t qb, uint32_t kst, uint32_t bar_s, int h, int npg)
{
    constexpr uint32_t id_s128 = umma_idesc_bf16(kRowsM, kBlockKeys, 0, 0);
    constexpr uint32_t id_s64 = umma_idesc_bf16(kRowsM, kPageSize, 0, 0);
    const uint32_t id = npg == 2 ? id_s128 : id_s64;
    const uint64_t a0 = umma_desc_sw128(qb + h * (2 * kRowsM * 128), 16, 1024);
    const uint64_t b0 = umma_desc_sw128(kst, 16, 1024);
    const uint32_t d = tmem + 256 * h;
    umma_bf16(d, a0, b0, id, false);
#pragma unroll
    for (int k = 1; k < kHeadDim / 16; ++k) {
        const uint32_t ao = ((k >> 2) * (kRowsM * 128) + (k & 3) * 32) >> 4;
        const uint32_t bo = ((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4;
        umma_bf16_acc(d, a0 + ao, b0 + bo, id);
    }
    umma_commit(bar_s + 8 * h);
}

// O_h (+)= P_h V for the npg pages of the V stage at `vs`; the first product
// of a run's first block overwrites O_h.
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t vs, int h, int npg, bool accumulate)
{
    constexpr uint32_t id_pv = umma_idesc_bf16(kRowsM, kHeadDim, 0, 1);
    const uint64_t b0 = umma_desc_sw128(vs, kHalfBytes, 1024);
    const uint32_t d = tmem + 256 * h + 128, a = tmem + 256 * h;
    umma_bf16_ts(d, a, b0, id_pv, accumulate);
#pragma unroll
    for (int k = 1; k < kPageSize / 16; ++k) umma_bf16_ts_acc(d, a + 8 * k, b0 + ((k * 2048) >> 4), id_pv);
    if (npg == 2) {  // the block's second page: one branch, not one per product
#pragma unroll
        for (int k = kPageSize / 16; k < kBlockKeys / 16; ++k)
            umma_bf16_ts_acc(d, a + 8 * k, b0 + ((k * 2048) >> 4), id_pv);
    }
}

// Every role runs its own unit loop through the same four CTA barriers per
// unit: (1) the unit the producer claimed is visible (and the producer has
// requested its Q, whose landing the issuer waits for on q_full), (2) the
// tile's tokens are loaded, (3) its runs are ready, (4) every product of the
// unit has completed (the epilogues waited for the last one), so that the next
// unit may rewrite Q and the token table.

// ---------------------------------------------------------------- producer (warp 8)
__device__ __forceinline__ void producer_role(const PfCtx& c, const PfParams& p, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, const CUtensorMap* tmQ, int first_claim,
                                              int lane)
{
    int q_load = 0;   // ring loads so far, across units
    int q_units = 0;  // units whose Q has been requested
    const uint64_t pol = l2_policy_evict_last();    // a prompt's tiles re-read the same pages
    const uint64_t pol_q = l2_policy_evict_first();  // each unit's Q is read once
    int claim = first_claim;  // the next unit, claimed before it is needed
    for (;;) {
        if (lane == 0) *c.sUnit = claim;
        __syncthreads();  // (1)
        const int u = *c.sUnit;
        if (u >= c.nunits || *c.abort_flag) break;
        const int g = u % p.kv_heads;
        if (lane == 0) {  // the unit's Q: the previous unit's products have all completed (barrier (4))
            int tile, run;
            item_of(c, p, u, tile, run);
            mbar_arrive_expect_tx(c.bar_q, kQBytes);
            for (int h = 0; h < kGroups; ++h)      // tokens 32h..32h+31 of the tile
                for (int half = 0; half < 2; ++half)  // dims 64 half ..
                    for (int j = 0; j < kGroup; ++j)  // query head g * 4 + j: rows 32j..32j+31
                        tma_load_3d(c.base + PfSmem::kQ + h * (2 * kRowsM * 128) + half * (kRowsM * 128) +
                                        j * (kHalfTok * 128),
                                    tmQ, 64 * half, g * kGroup + j, tile * kTileTok + kHalfTok * h, c.bar_q, pol_q);
        }
        ++q_units;
        __syncthreads();  // (2)
        {  // the unit's runs: all of the tile's, or the one its item names
            int tile, run;
            item_of(c, p, u, tile, run);
            const int nr = tile_runs(c.sPos[lane], c.sPos[lane + 32], c.sRow[lane], c.sRow[lane + 32],
                                     [&](int i, int row, int pages) {
                                         if (lane == 0 && (run < 0 || i == run)) {
                                             const int k = run < 0 ? i : 0;
                                             c.sRunRow[k] = row;
                                             c.sRunPages[k] = pages;
                                         }
                                     });
            if (lane == 0) *c.sNumRuns = run < 0 ? nr : (run < nr ? 1 : 0);
        }
        __syncthreads();  // (3)
        const int nruns = *c.sNumRuns;
        bool ok = true;
        for (int r = 0; r < nruns && ok; ++r) {
            const int row = c.sRunRow[r];
            const int n = c.sRunPages[r];
            for (int b0 = 0; b0 < n && ok; b0 += 32) {
                const int mine = (b0 + lane < n) ? page_of(p.table, p.pages, row, b0 + lane) : 0;
                for (int jj = 0; jj < min(32, n - b0) && ok; jj += 2) {
                    const int npg = min(2, n - b0 - jj);
                    const int pg0 = __shfl_sync(kAll, mine, jj);
                    const int pg1 = __shfl_sync(kAll, mine, jj + 1);
                    for (int kind = 0; kind < 2 && ok; ++kind) {  // the block's K, then its V
                        const int st = q_load % kPfStages;
                        if (q_load >= kPfStages)
                            ok = __all_sync(kAll, mbar_wait(c.bar_empty + 8 * st, ((q_load / kPfStages) - 1) & 1) &&
                                                      !*c.abort_flag);
                        if (!ok) break;
                        if (lane == 0) {
                            const CUtensorMap* tm = kind ? tmV : tmK;
                            const uint32_t fb = c.bar_full + 8 * st;
                            const uint32_t dst = c.base + PfSmem::kRing + st * kPfStageBytes;
                            mbar_arrive_expect_tx(fb, npg * 2 * kPageSize * 128);
                            for (int i = 0; i < npg; ++i) {
                                const int y = (i ? pg1 : pg0) * kPageSize;
                                tma_load_3d(dst + i * (kPageSize * 128), tm, 0, y, g, fb, pol);
                                tma_load_3d(dst + kHalfBytes + i * (kPageSize * 128), tm, 64, y, g, fb, pol);
                            }
                        }
                        ++q_load;
                        __syncwarp();
                    }
                }
            }
        }
        // the next unit is claimed once this one's last copy is out, about two blocks before
        // it ends: the counter's answer is back by then, and the units still go, longest
        // first, to the CTAs about to be free
        if (lane == 0) claim = atomicAdd(p.sched, 1);
        if (!ok && lane == 0) {
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            *c.abort_flag = 1;
            // let the copies in flight land before the CTA ends
            for (int k = max(0, q_load - kPfStages); k < q_load; ++k)
                mbar_wait(c.bar_full + 8 * (k % kPfStages), (k / kPfStages) & 1);
        }
        __syncthreads();  // (4)
    }
    // no copy in flight when the CTA ends (the issuer waited for every unit's Q unless it gave up)
    if (lane == 0 && q_units > 0) mbar_wait(c.bar_q, (q_units - 1) & 1);
}

// ---------------------------------------------------------------- MMA issuer (warp 9, one thread)
__device__ __forceinline__ void issuer_role(const PfCtx& c, const PfParams& p, int lane)
{
    const uint32_t qb = c.base + PfSmem::kQ, ring = c.base + PfSmem::kRing;
    const uint32_t tmem = c.tmem;
    int q_use = 0, it = 0, rc = 0;  // ring loads, blocks and runs so far, across units
    int uq = 0;                     // units so far (one Q copy each)
    for (;;) {
        __syncthreads();  // (1)
        if (*c.sUnit >= c.nunits || *c.abort_flag) break;
        __syncthreads();  // (2)
        tc_fence_before();
        __syncthreads();  // (3)
        tc_fence_after();
        const int nruns = *c.sNumRuns;
        if (lane == 0) {
            bool ok = mbar_wait_spin(c.bar_q, uq & 1) && !*c.abort_flag;  // the unit's Q has landed
            tc_fence_after();
            for (int r = 0; r < nruns && ok; ++r) {
                const int n = c.sRunPages[r];
                const int nb = (n + 1) / 2;
                {  // S_0(0), S_1(0)
                    const int st = q_use % kPfStages;
                    if (!mbar_wait_spin(c.bar_full + 8 * st, (q_use / kPfStages) & 1) || *c.abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kst = ring + st * kPfStageBytes;
                    issue_s(tmem, qb, kst, c.bar_s, 0, min(2, n));
                    issue_s(tmem, qb, kst, c.bar_s, 1, min(2, n));
                    umma_commit(c.bar_empty + 8 * st);
                }
                for (int b = 0; b < nb && ok; ++b) {
                    const int j = it + b;
                    const int vq = q_use + 2 * b + 1, vst = vq % kPfStages;
                    const int kq = vq + 1, kst = kq % kPfStages;
                    const int npg = min(2, n - 2 * b);
                    const bool more = b + 1 < nb;
                    if (!mbar_wait_spin(c.bar_full + 8 * vst, (vq / kPfStages) & 1) || *c.abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint32_t vs = ring + vst * kPfStageBytes;
                    for (int h = 0; h < kGroups; ++h) {
                        // O_h += P_h V_b once the softmax has written P_h (and, at a run's
                        // first block, the previous run's epilogue has read O_h)
                        if (!mbar_wait_spin(c.bar_p + 8 * h, j & 1) ||
                            (b == 0 && r > 0 && !mbar_wait_spin(c.bar_epi + 8 * h, (rc + r - 1) & 1)) ||
                            *c.abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(tmem, vs, h, npg, b > 0);
                        umma_commit(c.bar_o + 8 * h);
                        if (h == kGroups - 1) umma_commit(c.bar_empty + 8 * vst);
                        if (more) {  // S_h(b+1) over P_h(b), after the product that reads it
                            if (h == 0) {
                                if (!mbar_wait_spin(c.bar_full + 8 * kst, (kq / kPfStages) & 1) || *c.abort_flag) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                            }
                            issue_s(tmem, qb, ring + kst * kPfStageBytes, c.bar_s, h, min(2, n - 2 * b - 2));
                            if (h == kGroups - 1) umma_commit(c.bar_empty + 8 * kst);
                        }
                    }
                }
                it += nb;
                q_use += 2 * nb;
            }
            if (!ok) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                *c.abort_flag = 1;
            }
        }
        q_use = __shfl_sync(kAll, q_use, 0);
        it = __shfl_sync(kAll, it, 0);
        rc += nruns;
        ++uq;
        tc_fence_before();
        __syncthreads();  // (4)
        tc_fence_after();
    }
    if (lane == 0) {  // every product this thread issued has completed before the columns are freed
        umma_commit(c.bar_drain);
        mbar_wait_spin(c.bar_drain, 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- softmax group h (warps 4h..4h+3)
// Thread (warp w, lane) owns row 32 (w % 4) + lane of its group: query head
// 4g + w % 4 of token 32h + lane of the tile.
__device__ __forceinline__ void softmax_role(const PfCtx& c, const PfParams& p, int tid, int lane, int warp)
{
    const int h = warp >> 2, wq = warp & 3;
    const int tok = kHalfTok * h + lane;
    const uint32_t tl = c.tmem + ((uint32_t)(wq * 32) << 16) + 256 * h;  // S/P; O at +128
    int it = 0;  // blocks so far, across units
    for (;;) {
        __syncthreads();  // (1)
        const int u = *c.sUnit;
        if (u >= c.nunits || *c.abort_flag) break;
        const int g = u % p.kv_heads;
        int tile, run;
        item_of(c, p, u, tile, run);
        const int p0 = tile * kTileTok;
        if (tid < kTileTok) {  // the tile's tokens
            const int t = p0 + tid;
            const int len = t < p.P ? p.tok_len[t] : 0;
            c.sPos[tid] = len - 1;  // -1: not a token, or skipped
            c.sRow[tid] = len > 0 ? p.tok_row[t] : -1;
        }
        __syncthreads();  // (2)
        const int pos = c.sPos[tok];
        const int64_t qrow = ((int64_t)(p0 + tok) * p.heads + g * kGroup + wq) * kHeadDim;
        tc_fence_before();
        __syncthreads();  // (3)
        tc_fence_after();
        const int nruns = *c.sNumRuns;

        __nv_bfloat16* dst_row = p.out + qrow;
        bool ok = true;
        for (int r = 0; r < nruns && ok; ++r) {
            const int n = c.sRunPages[r];
            const int nb = (n + 1) / 2;
            const bool active = pos >= 0 && c.sRow[tok] == c.sRunRow[r];
            float m_used = -CUDART_INF_F, l = 0.f;
            for (int b = 0; b < nb; ++b) {
                const int j = it + b;
                // every exit decision is warp-wide: the tensor-memory accesses below are
                if (__any_sync(kAll, !mbar_wait_spin(c.bar_s + 8 * h, j & 1) || *c.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S of the block (a one-page block leaves columns 64..127 stale: the causal
                // mask removes them, every position of the run lies below its last page)
                const int lim = active ? pos - b * kBlockKeys : -1;  // keys c <= lim are visible
                const bool full = __all_sync(kAll, lim >= kBlockKeys - 1);
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32(tl, v0);
                tmem_ld32(tl + 32, v1);
                tmem_ld32(tl + 64, v2);
                tmem_ld32(tl + 96, v3);
                tmem_wait_ld_regs(v0);
                tmem_wait_ld_regs(v1);
                tmem_wait_ld_regs(v2);
                tmem_wait_ld_regs(v3);
                if (!full) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        if (k > lim) v0[k] = __float_as_uint(-CUDART_INF_F);
                        if (32 + k > lim) v1[k] = __float_as_uint(-CUDART_INF_F);
                        if (64 + k > lim) v2[k] = __float_as_uint(-CUDART_INF_F);
                        if (96 + k > lim) v3[k] = __float_as_uint(-CUDART_INF_F);
                    }
                }
                // row max, two new values per three-input max, four independent chains
                float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    mx4[0] = fmax3(mx4[0], __uint_as_float(v0[k]), __uint_as_float(v0[k + 1]));
                    mx4[1] = fmax3(mx4[1], __uint_as_float(v1[k]), __uint_as_float(v1[k + 1]));
                    mx4[2] = fmax3(mx4[2], __uint_as_float(v2[k]), __uint_as_float(v2[k + 1]));
                    mx4[3] = fmax3(mx4[3], __uint_as_float(v3[k]), __uint_as_float(v3[k + 1]));
                }
                const float mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
                // move the running max (rescaling O and l) only when this block raises it by > 8
                bool need = false;
                float alpha = 1.f;
                if (b == 0) {
                    m_used = mx;
                } else if (mx > m_used + kRescale) {
                    need = true;
                    alpha = exp2f(m_used - mx);
                }
                if (__any_sync(kAll, need)) {
                    // O must hold the previous block's product first
                    if (__any_sync(kAll, !mbar_wait_spin(c.bar_o + 8 * h, (j - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kHeadDim; k += 16) {
                        uint32_t v[16];
                        tmem_ld16(tl + 128 + k, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st16(tl + 128 + k, v);
                    }
                    tmem_wait_st();
                    if (need) {
                        l *= alpha;
                        m_used = mx;
                    }
                }
                // P = 2^(S - m) as bf16 pairs over the first half of S (a row with no key
                // yet has m = -inf: its p are all 0)
                const float msub = m_used == -CUDART_INF_F ? 0.f : m_used;
                // per pair of keys: one paired subtract, two exp2, one paired add to the
                // row sum, one paired conversion
                const uint64_t negm2 = f2_pack(-msub, -msub);
                uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};  // (+0.f, +0.f) pairs
                auto p_chunk = [&](const uint32_t (&v)[32], int cc) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float x0, x1;
                        f2_unpack(f2_add(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), negm2), x0, x1);
                        const float a = ex2_approx(x0), bb = ex2_approx(x1);
                        ps2[(e >> 1) & 3] = f2_add(ps2[(e >> 1) & 3], f2_pack(a, bb));
                        const __nv_bfloat162 ab = __floats2bfloat162_rn(a, bb);  // one paired conversion
                        pk[e / 2] = *reinterpret_cast<const uint32_t*>(&ab);
                    }
                    tmem_st16(tl + 16 * cc, pk);
                };
                p_chunk(v0, 0);
                p_chunk(v1, 1);
                p_chunk(v2, 2);
                p_chunk(v3, 3);
                {
                    float s[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) f2_unpack(ps2[k], s[2 * k], s[2 * k + 1]);
                    l += ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(c.bar_p + 8 * h);
            }
            if (!ok) break;
            // ---- epilogue of this row's pass: O / l for the active rows
            if (__any_sync(kAll, !mbar_wait_spin(c.bar_o + 8 * h, (it + nb - 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = active ? 1.f / l : 0.f;
#pragma unroll
            for (int k0 = 0; k0 < kHeadDim; k0 += 64) {
                uint32_t va[32], vb[32];
                tmem_ld32(tl + 128 + k0, va);
                tmem_ld32(tl + 128 + k0 + 32, vb);
                tmem_wait_ld_regs(va);
                tmem_wait_ld_regs(vb);
                if (active) {
#pragma unroll
                    for (int k = 0; k < 64; k += 8) {
                        const uint32_t* v = k < 32 ? va + k : vb + (k - 32);
                        uint32_t o4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 o2 = __floats2bfloat162_rn(__uint_as_float(v[2 * e]) * inv,
                                                                            __uint_as_float(v[2 * e + 1]) * inv);
                            o4[e] = *reinterpret_cast<const uint32_t*>(&o2);
                        }
                        *reinterpret_cast<uint4*>(dst_row + k0 + k) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(c.bar_epi + 8 * h);
            it += nb;
        }
        // skipped tokens of the tile: zero output
        if (ok && pos < 0 && p0 + tok < p.P) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
            for (int k = 0; k < kHeadDim / 8; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            *c.abort_flag = 1;
        }
        tc_fence_before();
        __syncthreads();  // (4)
        tc_fence_after();
    }
}

// ---------------------------------------------------------------- warps 10 and 11
__device__ __forceinline__ void idle_role(const PfCtx& c)
{
    for (;;) {
        __syncthreads();  // (1)
        if (*c.sUnit >= c.nunits || *c.abort_flag) break;
        __syncthreads();  // (2)
        __syncthreads();  // (3)
        __syncthreads();  // (4)
    }
}

// kSplit: a step whose rows' attention runs beside this grid (PfParams::split).
template <bool kSplit>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, PfParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    PfCtx c;
    c.base = (raw_base + 1023u) & ~1023u;
    c.sbase = smem_raw + (c.base - raw_base);
    const uint32_t bar0 = c.base + PfSmem::kBars;
    c.bar_full = bar0;
    c.bar_empty = bar0 + 8 * kPfStages;
    c.bar_s = bar0 + 16 * kPfStages;
    c.bar_p = c.bar_s + 8 * kGroups;
    c.bar_o = c.bar_p + 8 * kGroups;
    c.bar_epi = c.bar_o + 8 * kGroups;
    c.bar_drain = c.bar_epi + 8 * kGroups;
    c.bar_q = c.bar_drain + 8;
    uint32_t* sKey = reinterpret_cast<uint32_t*>(c.sbase + PfSmem::kSort);
    c.sKey = sKey;
    c.sPos = reinterpret_cast<int*>(c.sbase + PfSmem::kTok);
    c.sRow = c.sPos + kTileTok;
    c.sRunRow = reinterpret_cast<int*>(c.sbase + PfSmem::kRuns);
    c.sRunPages = c.sRunRow + kTileTok;
    c.sNumRuns = c.sRunPages + kTileTok;
    c.sUnit = c.sNumRuns + 1;
    c.abort_flag = reinterpret_cast<volatile int*>(c.sbase + PfSmem::kFlag);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < 2 * kPfStages; ++i) mbar_init(bar0 + 8 * i, 1);  // full (producer), empty (commit)
        for (int h = 0; h < kGroups; ++h) {
            mbar_init(c.bar_s + 8 * h, 1);
            mbar_init(c.bar_p + 8 * h, 4);
            mbar_init(c.bar_o + 8 * h, 1);
            mbar_init(c.bar_epi + 8 * h, 4);
        }
        mbar_init(c.bar_drain, 1);
        mbar_init(c.bar_q, 1);
        *c.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kIssuer) tmem_alloc(c.base + PfSmem::kTmemSlot, kTmemCols);
    if (warp == kProducer && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmQ);
    }
    pdl_wait();  // prep_kernel's appends, token table and zeroed unit counter
    // The kernel after this one in a step (the step rows' attention) reads only
    // what prep_kernel wrote: it may start on the SMs this grid leaves, and
    // waits for this grid before it ends.
    pdl_launch_dependents();
    // the producer's first unit is claimed now; the answer is needed after the sort
    int first_claim = 0;
    if (!kSplit && warp == kProducer && lane == 0) first_claim = atomicAdd(p.sched, 1);
    if (kSplit) {
        // The step rows' attention runs beside this grid: only the first prompt_sms(...)
        // CTAs go on, the others end here and leave their SMs to it (it derives the same
        // count from the same token lengths).  Warp w sums prompt_tile_cost over tiles
        // w, w + 12, ... (kTB tiles a round trip); every thread sums its rows' pages.
        unsigned long long* sSplit = reinterpret_cast<unsigned long long*>(c.sbase + PfSmem::kSplit);
        if (tid < 3) sSplit[tid] = 0ull;
        __syncthreads();
        constexpr int kWarps = kPfThreads / 32, kTB = 4;
        int64_t pc = 0, rp = 0;
        int pu = 0;
        for (int tb = warp; tb < p.ntiles; tb += kTB * kWarps) {
            int m[kTB][2];
#pragma unroll
            for (int b = 0; b < kTB; ++b)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tok = (tb + b * kWarps) * kTileTok + lane + 32 * i;
                    m[b][i] = (tb + b * kWarps < p.ntiles && tok < p.P) ? p.tok_len[tok] : 0;
                }
#pragma unroll
            for (int b = 0; b < kTB; ++b) {
                const int mx = (int)__reduce_max_sync(kAll, (uint32_t)max(max(m[b][0], m[b][1]), 0));
                pc += prompt_tile_cost(mx, p.kv_heads);
                pu += mx > 0 ? p.kv_heads : 0;
            }
        }
        for (int r = tid; r < p.steps; r += kPfThreads) {
            const int len = p.tok_len[p.P + r];
            rp += len > 0 ? (len + kPageSize - 1) / kPageSize : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) rp += __shfl_xor_sync(kAll, rp, o);
        if (lane == 0) {
            if (pc) atomicAdd(&sSplit[0], (unsigned long long)pc);
            if (pu) atomicAdd(&sSplit[1], (unsigned long long)pu);
            if (rp) atomicAdd(&sSplit[2], (unsigned long long)rp);
        }
        tc_fence_before();
        __syncthreads();
        const int keep = prompt_sms((int64_t)sSplit[0], kSplitRowPage * p.kv_heads * (int64_t)sSplit[2],
                                    (int)sSplit[1], p.sms);
        if ((int)blockIdx.x >= keep) {  // this CTA ends here, its tensor memory freed first
            if (warp == kIssuer) {
                tc_fence_after();
                tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(c.sbase + PfSmem::kTmemSlot), kTmemCols);
            }
            return;
        }
        if (warp == kProducer && lane == 0) first_claim = atomicAdd(p.sched, 1);
    }

    // ---- work items: the runs of every tile (a tile with none is one empty item,
    // so that its skipped tokens still get their zero output), in decreasing order
    // of pages, ties in token order
    const int ntiles = p.ntiles;
    int* sNItems = c.sUnit + 1;
    if (tid == 0) *sNItems = 0;
    __syncthreads();
    if (ntiles <= kMaxSortTiles) {
        // warp w takes tiles w, w + 12, ...: the lengths and rows of kScanBatch of
        // them are loaded before the first is looked at (one memory latency a batch)
        constexpr int kWarps = kPfThreads / 32, kScanBatch = 4;
        for (int t0 = warp; t0 < ntiles; t0 += kScanBatch * kWarps) {
            int lens[kScanBatch][2], rows[kScanBatch][2];
#pragma unroll
            for (int bt = 0; bt < kScanBatch; ++bt)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tok = (t0 + bt * kWarps) * kTileTok + lane + 32 * i;
                    const bool in = t0 + bt * kWarps < ntiles && tok < p.P;
                    lens[bt][i] = in ? p.tok_len[tok] : 0;
                    rows[bt][i] = in ? p.tok_row[tok] : -1;
                }
#pragma unroll
            for (int bt = 0; bt < kScanBatch; ++bt) {
            const int t = t0 + bt * kWarps;
            if (t >= ntiles) break;  // the same for the whole warp
            int pos2[2], row2[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                pos2[i] = lens[bt][i] - 1;
                row2[i] = lens[bt][i] > 0 ? rows[bt][i] : -1;
            }
            auto add = [&](int run, int pages) {
                if (lane == 0) {
                    const int idx = atomicAdd(sNItems, 1);
                    if (idx < kMaxSortTiles)
                        sKey[idx] = ((uint32_t)pages << kKeyPagesShift) |
                                    ((uint32_t)((kMaxSortTiles - 1) - t) << kKeyTileShift) | (uint32_t)(63 - run);
                }
            };
            const int nr = tile_runs(pos2[0], pos2[1], row2[0], row2[1], [&](int i, int, int pages) { add(i, pages); });
            if (nr == 0) add(0, 0);
            }
        }
    } else if (tid == 0) {
        *sNItems = kMaxSortTiles + 1;
    }
    __syncthreads();
    const int nitems = *sNItems;
    c.sorted = nitems <= kMaxSortTiles;
    c.nunits = (c.sorted ? nitems : ntiles) * p.kv_heads;
    if (c.sorted && nitems <= kPfThreads) {
        // one key a thread; keys are distinct (each names its tile and run), so a
        // key's place in decreasing order is the number of larger keys
        uint32_t key = 0;
        int rank = 0;
        if (tid < nitems) {
            key = sKey[tid];
            for (int i = 0; i < nitems; ++i) rank += sKey[i] > key;
        }
        __syncthreads();
        if (tid < nitems) sKey[rank] = key;
    } else if (c.sorted) {
        int n2 = 1;
        while (n2 < nitems) n2 <<= 1;
        for (int i = nitems + tid; i < n2; i += kPfThreads) sKey[i] = 0;
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) {  // bitonic sort, descending
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < n2; i += kPfThreads) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const uint32_t a = sKey[i], b = sKey[ixj];
                        if (((i & k) == 0) ? (a < b) : (a > b)) {
                            sKey[i] = b;
                            sKey[ixj] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *reinterpret_cast<volatile uint32_t*>(c.sbase + PfSmem::kTmemSlot);

    if (warp >= kProducer) {
        regs_dec<kRegsOther>();
        if (warp == kProducer)
            producer_role(c, p, &tmK, &tmV, &tmQ, first_claim, lane);
        else if (warp == kIssuer)
            issuer_role(c, p, lane);
        else
            idle_role(c);
    } else {
        regs_inc<kRegsSoftmax>();
        softmax_role(c, p, tid, lane, warp);
    }
}

}  // namespace

cudaError_t configure_prefill()
{
    // The kernel moves registers between its warpgroups assuming it is launched
    // with exactly kRegsLaunch per thread; refuse to run it with any other count.
    cudaFuncAttributes fa;
    for (auto k : {prefill_kernel<false>, prefill_kernel<true>}) {
        cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != (int)kRegsLaunch) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem::kAlloc);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_prefill(const pkv_pool* pool, const StepArgs& a, const Plan& plan, int ctas, bool split,
                           cudaStream_t s)
{
    PfParams p;
    p.tok_len = reinterpret_cast<const int32_t*>(a.ws + plan.off_len);
    p.tok_row = reinterpret_cast<const int32_t*>(a.ws + plan.off_row);
    p.table = a.table;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.sched = reinterpret_cast<int32_t*>(a.ws + plan.off_sched);
    p.err = pool->err;
    p.P = a.P;
    p.pages = a.pages;
    p.heads = pool->cfg.heads;
    p.kv_heads = pool->cfg.kv_heads;
    p.ntiles = (a.P + kTileTok - 1) / kTileTok;
    p.split = split && a.steps > 0 ? 1 : 0;
    p.steps = a.steps;
    p.sms = pool->num_sms;
    // the prompt tokens' queries prep_kernel prepared in the workspace
    CUtensorMap tmQ;
    if (!make_tmap_heads(&tmQ, a.ws + plan.off_qhat, p.heads, a.P)) return cudaErrorInvalidValue;
    const int units = p.ntiles * p.kv_heads;
    const int grid = ctas < units ? ctas : units;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = PfSmem::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.split ? cudaLaunchKernelEx(&cfg, prefill_kernel<true>, pool->tmap_k, pool->tmap_v, tmQ, p)
                   : cudaLaunchKernelEx(&cfg, prefill_kernel<false>, pool->tmap_k, pool->tmap_v, tmQ, p);
}

}  // namespace pkv
