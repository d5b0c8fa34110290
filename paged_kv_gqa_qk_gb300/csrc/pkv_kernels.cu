// Kernels of the paged-KV decode step (sm_103a).
//
//   attn_kernel     persistent split-KV attention.  The work is the sequence
//                   of (token, kv head, page) triples; each CTA streams an
//                   equal slice of most of it, whatever the mix of row
//                   lengths, then claims small chunks of the rest as it
//                   finishes (split_of).  A producer warp streams the pages
//                   through a shared-memory ring with TMA; four consumer warps
//                   run QK^T and PV on mma.sync tensor cores with an online
//                   softmax.  In decode mode the kernel also does the per-token
//                   work before attention: it validates each row, norms and
//                   ropes the query heads it attends with, and appends the
//                   row's new k and v (see attn_kernel).
//   combine_kernel  log-sum-exp merge of the pieces of a (token, kv head) that
//                   several CTAs shared; zero outputs for skipped tokens.
//   prep_kernel     step mode only: validates every token and appends all k/v
//                   before any attention (the prompt tokens of a chunk read
//                   each other's keys), and writes each prompt token's query
//                   heads, normed, roped and scaled, for the prompt attention.
//
// Source of the computation: qwen3-8b Nest files, src/attention.linnet,
// GroupedQueryAttention.decode_paged / step_paged (q_norm/k_norm -> rope_rows
// -> page_slots + write_tokens -> paged_attention), src/norm.linnet (RmsNorm,
// eps 1e-6), src/rope.linnet (rotate-half tables, base 1e6).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "pkv_rope.cuh"

namespace pkv {

// =====================================================================================
// prep_kernel (step mode): validate every token, append every token's k and v,
// prepare the prompt tokens' queries
// =====================================================================================
constexpr int kPrepWarps = 4;                 // warps of a token's CTA
constexpr int kKvPre = 8 / kPrepWarps;        // kv heads a warp loads before the first use (of 8)
struct PrepParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* qw;
    const __nv_bfloat16* kw;
    const int32_t* positions;       // [P]
    const int32_t* prow;            // [P]
    const int32_t* slots;           // [P] or null
    const int32_t* step_positions;  // [rows]
    const int32_t* table;           // [rows][pages], or null: contiguous rows
    int P, rows, pages, num_pages, max_seq, heads, kv_heads, rot;
    int64_t num_slots;
    float eps;
    const float2* rope_hi;          // (cos, sin) [max_seq][64], fp32 nearest to the double values
    const float2* rope_lo;          // the double values minus rope_hi, in fp32
    __nv_bfloat16* K;               // [kv_heads][num_slots][128]
    __nv_bfloat16* V;
    __nv_bfloat16* q_hat;           // [P][heads][128]: the prompt attention's queries
    int32_t* tok_len;               // [tokens]  attended length, 0 = skip
    int32_t* tok_row;               // [tokens]  table row
    int32_t* sched;                 // work-unit counter of the prompt attention, zeroed here
    uint32_t* err;
};

// One CTA (kPrepWarps warps) per token; warp w appends kv heads w, w + 4, ...
// and, for a prompt token, prepares its query heads w, w + 4, ...  The loads
// that depend only on the token index (its q, k and v) go out first, the ones
// that need its row and position (the table entries, the slot, the RoPE row)
// next, all before the first use, so that the token costs about two memory
// latencies.  (Four warps a token measured faster than one, two or eight: the
// per-warp chain of norms outweighs the residency fewer threads would give.)
__global__ void __launch_bounds__(32 * kPrepWarps) prep_kernel(PrepParams p)
{
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // first the loads that depend on nothing but t: the token's k and v for
    // this warp's first kv heads, a prompt token's first query heads of this
    // warp and the q weights
    uint2 kraw[kKvPre] = {}, vraw[kKvPre] = {};
#pragma unroll
    for (int i = 0; i < kKvPre; ++i) {
        const int g = warp + kPrepWarps * i;
        if (g < p.kv_heads) {
            const int64_t src = ((int64_t)t * p.kv_heads + g) * kHeadDim + 4 * lane;
            kraw[i] = *reinterpret_cast<const uint2*>(p.k + src);
            vraw[i] = *reinterpret_cast<const uint2*>(p.v + src);
        }
    }
    constexpr int kQPre = 32 / kPrepWarps;
    const bool prompt = t < p.P;
    uint2 qraw[kQPre] = {};
    float wq[4] = {};
    if (prompt) {
#pragma unroll
        for (int i = 0; i < kQPre; ++i)
            if (warp + kPrepWarps * i < p.heads)
                qraw[i] = *reinterpret_cast<const uint2*>(p.q + ((int64_t)t * p.heads + warp + kPrepWarps * i) * kHeadDim + 4 * lane);
        unpack4(*reinterpret_cast<const uint2*>(p.qw + 4 * lane), wq);
    }

    int row, pos;
    bool active = true;
    if (t < p.P) {
        row = p.prow[t];
        pos = p.positions[t];
    } else {
        row = t - p.P;
        pos = p.step_positions[row];
        active = pos != -1;  // -1: the row takes no step
    }
    uint32_t e = 0;
    if (active) {
        if (row < 0 || row >= p.rows)
            e = PKV_DEVERR_ROW;
        else if (pos < 0 || pos >= p.max_seq || pos >= p.pages * kPageSize)
            e = PKV_DEVERR_POSITION;
    }
    const bool inrange = active && !e;
    // every page the token will read must be a pool page
    int bad = 0;
    const int npg = inrange ? pos / kPageSize + 1 : 0;
    for (int i = tid; i < npg; i += blockDim.x) {
        const int id = page_of(p.table, p.pages, row, i);
        bad |= (id < 0 || id >= p.num_pages);
    }
    int64_t slot = 0;
    if (inrange) {
        if (t < p.P && p.slots)
            slot = p.slots[t];
        else
            slot = (int64_t)page_of(p.table, p.pages, row, pos / kPageSize) * kPageSize + pos % kPageSize;
    }
    // the token's RoPE row and the k weights
    const int pc = inrange ? pos : 0;
    float2 rh[4], rl[4];
    {
        const int f0 = krope(lane, p.rot).f0;
        const float4* h4 = reinterpret_cast<const float4*>(p.rope_hi + (int64_t)pc * kRopeHalf + f0);
        const float4* l4 = reinterpret_cast<const float4*>(p.rope_lo + (int64_t)pc * kRopeHalf + f0);
        const float4 a = h4[0], b = h4[1], c = l4[0], d = l4[1];
        rh[0] = make_float2(a.x, a.y), rh[1] = make_float2(a.z, a.w), rh[2] = make_float2(b.x, b.y),
        rh[3] = make_float2(b.z, b.w);
        rl[0] = make_float2(c.x, c.y), rl[1] = make_float2(c.z, c.w), rl[2] = make_float2(d.x, d.y),
        rl[3] = make_float2(d.z, d.w);
    }
    float wk[4];
    unpack4(*reinterpret_cast<const uint2*>(p.kw + 4 * lane), wk);

    bad = __syncthreads_or(bad);
    if (inrange && bad) e = PKV_DEVERR_PAGE;
    if (inrange && !e && t < p.P && p.slots && (slot < 0 || slot >= p.num_slots)) e = PKV_DEVERR_SLOT;
    if (tid == 0) {
        if (t == 0) *p.sched = 0;
        const bool ok = active && !e;
        p.tok_len[t] = ok ? pos + 1 : 0;
        p.tok_row[t] = ok ? row : 0;
        if (e) atomicOr(p.err, e);
    }
    if (prompt) {
        // the prompt attention's queries: QK-norm + RoPE (fp32 cos, sin), times
        // kQScale, in bf16; zero for a skipped token
        const bool ok = active && !e;
        auto prep_q = [&](int hq, uint2 raw) {
            uint2 r = make_uint2(0u, 0u);
            if (ok) {
                const float4 y = norm_rope_q_regs(raw, wq, rh, p.eps, lane, p.rot);
                const float ys[4] = {y.x * kQScale, y.y * kQScale, y.z * kQScale, y.w * kQScale};
                r = pack4(ys);
            }
            *reinterpret_cast<uint2*>(p.q_hat + ((int64_t)t * p.heads + hq) * kHeadDim + 4 * lane) = r;
        };
#pragma unroll
        for (int i = 0; i < kQPre; ++i)
            if (warp + kPrepWarps * i < p.heads) prep_q(warp + kPrepWarps * i, qraw[i]);
        for (int hq = warp + kPrepWarps * kQPre; hq < p.heads; hq += kPrepWarps)
            prep_q(hq, *reinterpret_cast<const uint2*>(p.q + ((int64_t)t * p.heads + hq) * kHeadDim + 4 * lane));
    }
    if (!active || e) return;

    auto append = [&](int g, uint2 kr, uint2 vr) {
        const int64_t dst = ((int64_t)g * p.num_slots + slot) * kHeadDim + 4 * lane;
        *reinterpret_cast<uint2*>(p.K + dst) = norm_rope_k_regs(kr, wk, rh, rl, p.eps, lane, p.rot);
        *reinterpret_cast<uint2*>(p.V + dst) = vr;  // v is written as given
    };
#pragma unroll
    for (int i = 0; i < kKvPre; ++i)
        if (warp + kPrepWarps * i < p.kv_heads) append(warp + kPrepWarps * i, kraw[i], vraw[i]);
    for (int g = warp + kPrepWarps * kKvPre; g < p.kv_heads; g += kPrepWarps) {
        const int64_t src = ((int64_t)t * p.kv_heads + g) * kHeadDim + 4 * lane;
        append(g, *reinterpret_cast<const uint2*>(p.k + src), *reinterpret_cast<const uint2*>(p.v + src));
    }
}

cudaError_t launch_prep(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s)
{
    PrepParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.k = static_cast<const __nv_bfloat16*>(a.k);
    p.v = static_cast<const __nv_bfloat16*>(a.v);
    p.qw = static_cast<const __nv_bfloat16*>(a.q_norm_w);
    p.kw = static_cast<const __nv_bfloat16*>(a.k_norm_w);
    p.positions = a.positions;
    p.prow = a.prow;
    p.slots = a.slots;
    p.step_positions = a.step_positions;
    p.table = a.table;
    p.P = a.P;
    p.rows = a.rows;
    p.pages = a.pages;
    p.num_pages = pool->num_pages;
    p.max_seq = pool->cfg.max_seq;
    p.heads = pool->cfg.heads;
    p.kv_heads = pool->cfg.kv_heads;
    p.rot = pool->cfg.rotary_dim > 0 ? pool->cfg.rotary_dim : kHeadDim;
    p.num_slots = pool->num_slots;
    p.eps = static_cast<float>(pool->cfg.eps);
    p.rope_hi = pool->rope_hi;
    p.rope_lo = pool->rope_lo;
    p.K = static_cast<__nv_bfloat16*>(pool->k);
    p.V = static_cast<__nv_bfloat16*>(pool->v);
    p.q_hat = reinterpret_cast<__nv_bfloat16*>(a.ws + plan.off_qhat);
    p.tok_len = reinterpret_cast<int32_t*>(a.ws + plan.off_len);
    p.tok_row = reinterpret_cast<int32_t*>(a.ws + plan.off_row);
    p.sched = reinterpret_cast<int32_t*>(a.ws + plan.off_sched);
    p.err = pool->err;
    prep_kernel<<<a.P + a.steps, 32 * kPrepWarps, 0, s>>>(p);
    return cudaGetLastError();
}

// =====================================================================================
// attn_kernel: persistent split-KV attention with a static + dynamic work split
// =====================================================================================
//
// Work order.  Tokens in order; within a token its kv heads; within a kv head
// its pages 0..npg-1: unit u = t*G + g covers global pages
// [G*pre[t] + g*npg[t], + npg[t]) with pre the exclusive prefix of npg over
// tokens, T = G*sum(npg) pages in all.  split_of cuts the sequence into
// intervals: a static slice per CTA (CTAs beyond min(C, T) idle), then chunks
// the CTAs claim from a counter as they finish.  The piece of a unit inside one
// interval is a segment.  A unit wholly inside one interval is written out
// directly; otherwise each piece leaves a partial (O/l and the base-2
// log-sum-exp, for the 4 query heads) at index u + i for interval i -- unique,
// because units and intervals both increase along the sequence -- and
// combine_kernel merges them in interval order, whichever CTA streamed each.
// After its last range the producer sends a ring item without data that stops
// the consumers.
//
// Per page, consumer warp w takes positions 16w..16w+15:
//   QK^T:  S[16 pos][8 cols] = K_tile[16][128] * Qb[128][8]
//          cols 0-3 = bf16 head of q (heads 4g..4g+3, scaled by log2(e)/sqrt(128)),
//          cols 4-7 = bf16 of the remainder; S = col h + col h+4 keeps ~16 bits of q.
//   PV:    O^T[128][8] += V_tile^T[128][16 pos] * Pb[16 pos][8]
//          cols 0-3 = bf16(p), cols 4-7 = bf16(p - bf16(p)); O = col h + col h+4.
// Softmax state (running max m, sum l, per head, base 2) is per warp; the four
// warps are merged through shared memory, in a fixed order, at the end of
// each segment.
//
// Decode mode appends each row's new k and v: the CTA holding a unit's last
// page receives the row's raw k/v with the segment, and the consumer warp
// that owns the new slot's position norms and ropes k, writes it and v into
// its staged copy of the page and to the pool.  Each (row, kv head) slot is
// read only by that row (a documented condition of pkv_decode), so no other
// CTA waits for the write.
// B fragments of q for one head: the dims 16 ks + 2 tig + {0, 1, 8, 9} (ks < 8)
// this lane holds, normed (xr raw, wq2 weights, inv = 1/rms times the score
// scale) and rotated with the pairs (d, d + 16 HK) of a 32 HK-dim rotation
// (rpf: the position's (cos, sin) table), dims from 32 HK up unrotated; split
// into a bf16 head (prt 0) or the bf16 of its remainder (prt 1).
template <int HK>
__device__ __forceinline__ void q_prep(const uint32_t (&xr)[8][2], const uint32_t (&wq2)[8][2], const float2* rpf,
                                       float inv, int tig, int prt, uint32_t (&bq)[8][2])
{
    auto part = [&](const float (&y)[4], uint32_t (&dst)[2]) {
        __nv_bfloat16 h[4], t[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) split_bf16(y[k], h[k], t[k]);
        dst[0] = prt ? pack_bf16(t[0], t[1]) : pack_bf16(h[0], h[1]);
        dst[1] = prt ? pack_bf16(t[2], t[3]) : pack_bf16(h[2], h[3]);
    };
    auto u_of = [&](uint32_t x, uint32_t w, int b) {
        return __uint_as_float(b ? (x & 0xffff0000u) : (x << 16)) * __uint_as_float(b ? (w & 0xffff0000u) : (w << 16));
    };
#pragma unroll
    for (int ks = 0; ks < HK; ++ks) {  // dims d (ks) and their partners d + 16 HK (ks + HK)
        float ylo[4], yhi[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int d = 16 * ks + 2 * tig + 8 * e + b;  // < 16 HK
                const float ul = u_of(xr[ks][e], wq2[ks][e], b), uh = u_of(xr[ks + HK][e], wq2[ks + HK][e], b);
                const float2 cs = rpf[d];
                ylo[2 * e + b] = inv * (ul * cs.x - uh * cs.y);  // y[d]         = u[d] cos - u[d+16HK] sin
                yhi[2 * e + b] = inv * (uh * cs.x + ul * cs.y);  // y[d + 16 HK] = u[d+16HK] cos + u[d] sin
            }
        }
        part(ylo, bq[ks]);
        part(yhi, bq[ks + HK]);
    }
#pragma unroll
    for (int ks = 2 * HK; ks < 8; ++ks) {  // dims RoPE leaves as they are
        float y[4];
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int b = 0; b < 2; ++b) y[2 * e + b] = inv * u_of(xr[ks][e], wq2[ks][e], b);
        part(y, bq[ks]);
    }
}

// B fragments of q for one head, from q already normed and roped (fp32, the
// head's 128 dims at qf; pkv_qkv_proj_append's output): the dims
// 16 ks + 2 tig + {0, 1, 8, 9} of this lane, times the score scale, split into
// a bf16 head (prt 0) or the bf16 of its remainder (prt 1).
__device__ __forceinline__ void q_from_hat(const float* qf, float scale, int tig, int prt, uint32_t (&bq)[8][2])
{
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const float2 lo = *reinterpret_cast<const float2*>(qf + 16 * ks + 2 * tig);
        const float2 hi = *reinterpret_cast<const float2*>(qf + 16 * ks + 2 * tig + 8);
        const float y[4] = {lo.x * scale, lo.y * scale, hi.x * scale, hi.y * scale};
        __nv_bfloat16 h[4], t[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) split_bf16(y[k], h[k], t[k]);
        bq[ks][0] = prt ? pack_bf16(t[0], t[1]) : pack_bf16(h[0], h[1]);
        bq[ks][1] = prt ? pack_bf16(t[2], t[3]) : pack_bf16(h[2], h[3]);
    }
}

struct AttnParams {
    const __nv_bfloat16* q;   // [ntok][heads][128] projected q (normed + roped here)
    const float* qhat;        // prepared mode: [ntok][heads][128] q already normed + roped, fp32
    const __nv_bfloat16* k;   // [ntok][kv_heads][128]  (decode mode: appended here)
    const __nv_bfloat16* v;
    const __nv_bfloat16* qw;
    const __nv_bfloat16* kw;
    const int32_t* positions; // decode mode: [ntok], token t is table row t
    const int32_t* tok_len;   // step mode: [ntok] from prep_kernel, 0 = skip
    const int32_t* tok_row;   // step mode: [ntok]
    const int32_t* table;     // [rows][pages]
    const float2* rope_hi;    // (cos, sin) [max_seq][64], fp32 nearest to the double values
    const float2* rope_lo;    // the double values minus rope_hi, in fp32 (k only)
    __nv_bfloat16* K;         // pool
    __nv_bfloat16* V;
    __nv_bfloat16* out;       // [ntok][heads][128]
    float* part_o;            // [U + C (1 + kDynChunksPerCta)][4][128]
    float* part_lse;          // [U + C (1 + kDynChunksPerCta)][4]
    uint32_t* claim;          // chunk counter, zero at launch
    int32_t* prefix;          // [ntok + 2], written by CTA 0 for combine_kernel: prefix, total, resident CTAs
    int32_t* unit_ok;         // [U], by the CTA holding each unit's first page: 0 invalid, 1 cut, 2 written out
    uint32_t* err;
    int ntok, pages, num_pages, max_seq, heads, kv_heads, decode_mode, rot;
    int rows;                 // table rows (for the neighbouring-row comparison of shared pages)
    int prepared;             // decode mode with q prepared and k/v appended beforehand (pkv_decode_appended)
    int late_wait;            // step mode after the prompt attention: see the launch wait in attn_kernel
    int64_t num_slots;
    float eps;
    uint64_t wait_ns;         // limit of the ring and group waits (the final drain always allows kWaitLimitNs)
    int prompt_P;             // step mode: the call's prompt tokens (their lengths precede tok_len), else 0
    int sms, ctas_per_sm;     // the device's SMs, and this kernel's resident CTAs per SM
};

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = 4 * 8192;  // K lo, K hi, V lo, V hi
// Per stage, for a segment's first page: raw q of the 4 heads (1 KiB) and the
// (cos, sin) hi parts of the token's position (512 B); when the segment holds
// the row's new slot (decode mode) also the lo parts (512 B) and the raw k
// and v (256 B each).
constexpr int kSideBytes = 2560;
constexpr int kSideQ = 0, kSideRopeHi = 1024, kSideRopeLo = 1536, kSideK = 2048, kSideV = 2304;

constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagValid = 4, kFlagComplete = 8, kFlagHasLast = 16,
              kFlagAppend = 32, kFlagStop = 64;

template <int kStages>
struct AttnSmem {
    static constexpr int kSide = kStages * kStageBytes;
    static constexpr int kM = kSide + kStages * kSideBytes;  // float [4 warps][4 heads]
    static constexpr int kL = kM + 64;                        // float [4][4]
    static constexpr int kMeta = kL + 64;                     // int4 [stages][2]
    // int [32]: per warp the page sums [0, 8), the largest unit [8, 16) and the tokens
    // with pages [16, 24); the first token of the CTA's slice and its prefix at 24, 25
    static constexpr int kScan = kMeta + kStages * 32;
    static constexpr int kSum = kScan + 128;                  // int [threads] first token, int [threads] prefix
    static_assert(kAttnThreads / 32 <= 8, "a warp's entries of the scan fit");
    // int [threads] each: pages, length and table row per token (read by the whole-unit split)
    static constexpr int kTokN = kSum + 2 * kAttnThreads * 4;
    static constexpr int kTokLen = kTokN + kAttnThreads * 4;
    static constexpr int kTokRow = kTokLen + kAttnThreads * 4;
    static constexpr int kSplit = kTokRow + kAttnThreads * 4;  // per warp: int64 prompt cost [8], int units [8]
    static constexpr int kW = kSplit + 8 * 8 + 8 * 4;         // bf16 q_norm_w [128], k_norm_w [128]
    static constexpr int kBars = kW + 512;                    // u64 full[S], empty[S], group
    static constexpr int kFlag = kBars + 8 * (2 * kStages + 1);  // int abort, items issued, stop item sent
    static constexpr int kBytes = kFlag + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
};

// The work split.  Global pages [0, T) are cut into intervals: first Ce =
// min(C, T) static slices of the first S pages, slice c = [c*S/Ce, (c+1)*S/Ce)
// for CTA c; then, when there are two CTAs or more and at least
// kDynMinPagesPerCta pages per CTA, a quarter of the pages in ND chunks of Q
// pages, chunk k = [S + kQ, S + (k+1)Q),
// which the CTAs claim from a counter once their slice is done.  The CTAs'
// streaming rates differ by some 10-20% (the same pages take longer on some
// SMs), so equal static slices alone end at different times; the chunks let
// the fast CTAs take over the rest.  Q is 4 pages, or more where that keeps
// ND <= kDynChunksPerCta * Ce (the partial slots of the workspace).  (Smaller
// chunks cost more than they balance: each is a segment of its own, with the
// q preparation at its start and the merge and partial write at its end.)
constexpr int kDynMinPagesPerCta = 8;
constexpr int kDynChunkPages = 4;
constexpr int kClaimAhead = 2;  // pages of a range still to issue when the next chunk is claimed

struct Split {
    int64_t S;  // pages in static slices
    int Ce;     // static slices (CTAs with work)
    int ND;     // chunks after them
    int Q;      // pages per chunk
    int whole;  // whole units instead (see whole_split): Ce first units, then ND claimed ones
};

__device__ __forceinline__ Split split_of(int64_t T, int C)
{
    Split sp;
    sp.Ce = (int)min((int64_t)C, T);
    sp.S = T;
    sp.ND = 0;
    sp.Q = kDynChunkPages;
    sp.whole = 0;
    if (sp.Ce > 1 && T >= (int64_t)kDynMinPagesPerCta * sp.Ce) {
        const int64_t dyn = T / 4, cap = (int64_t)kDynChunksPerCta * sp.Ce;
        sp.Q = (int)max((int64_t)kDynChunkPages, (dyn + cap - 1) / cap);
        sp.ND = (int)(dyn / sp.Q);
        sp.S = T - (int64_t)sp.ND * sp.Q;
    }
    return sp;
}

// The whole-unit split, for calls of short rows: when every token has a thread
// of the prologue (ntok <= kAttnThreads), no unit is longer than
// kWholeMaxPages and the longest is within 5/4 of a CTA's share of the pages,
// no unit is cut at all.  The units go out longest first (tokens ordered by
// their page count, ties by index; a token's kv heads in order): CTA c takes
// unit c, and the rest are claimed one at a time from the chunk counter.  Each
// unit is then one segment, written out by the CTA that streams it, and the
// last units handed out are the shortest; with slices and chunks a call of
// short rows pays several segments a CTA (a preparation of q at the start of
// each, a merge and a partial at its end) and a tail of a whole chunk.
constexpr int kWholeMaxPages = 16;

__device__ __forceinline__ bool whole_units(int ntok, int nmax, int64_t T, int C)
{
    return ntok <= kAttnThreads && nmax <= kWholeMaxPages && 4 * (int64_t)nmax * C <= 5 * T;
}

__device__ __forceinline__ Split whole_split(int units, int C)
{
    Split sp;
    sp.Ce = min(C, units);
    sp.ND = units - sp.Ce;
    sp.S = 0;
    sp.Q = 0;
    sp.whole = 1;
    return sp;
}

// Slice c of C (C <= T) covers pages [c*T/C, (c+1)*T/C); the slice holding page x.
__device__ __forceinline__ int cta_of(int64_t x, int64_t T, int C)
{
    int c = (int)(x * C / T);
    while (c + 1 < C && (int64_t)(c + 1) * T / C <= x) ++c;
    while (c > 0 && (int64_t)c * T / C > x) --c;
    return c;
}

// The interval (static slice or chunk) holding global page x < T.
__device__ __forceinline__ int interval_of(int64_t x, const Split& sp)
{
    return x < sp.S ? cta_of(x, sp.S, sp.Ce) : sp.Ce + (int)((x - sp.S) / sp.Q);
}

// What token t's page count comes from: its position (decode mode) or its length.
__device__ __forceinline__ int tok_value(const AttnParams& p, int t)
{
    return p.decode_mode ? p.positions[t] : p.tok_len[t];
}

__device__ __forceinline__ int npg_from(const AttnParams& p, int v)
{
    if (p.decode_mode) return (v >= 0 && v < p.max_seq && v < p.pages * kPageSize) ? v / kPageSize + 1 : 0;
    return v > 0 ? (v + kPageSize - 1) / kPageSize : 0;
}

__device__ __forceinline__ int npg_of(const AttnParams& p, int t) { return npg_from(p, tok_value(p, t)); }

__device__ __forceinline__ void token_info(const AttnParams& p, int t, int& row, int& len)
{
    if (p.decode_mode) {
        row = t;
        len = p.positions[t] + 1;
    } else {
        row = p.tok_row[t];
        len = p.tok_len[t];
    }
}

// The four consumer warps meet at an mbarrier (bounded wait, unlike bar.sync);
// the result is the same on every lane of the warp.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, int lane, uint64_t limit_ns)
{
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = __all_sync(kFull, mbar_wait_spin(bar, phase & 1, limit_ns));
    ++phase;
    return ok;
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Warp-wide: the token t holding global page x (x < T) and its prefix pre[t],
// from the per-thread summaries of the prologue (first token and prefix of each
// thread's run of tokens) and one pass over that run.
__device__ __forceinline__ void find_token(const AttnParams& p, const int* sT0, const int* sP0, int64_t x, int lane,
                                           int& t_out, int& pre_out)
{
    const int G = p.kv_heads;
    int lo = 0, hi = kAttnThreads - 1;
    while (lo < hi) {  // last run whose prefix starts at or before x
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)G * sP0[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    int t = sT0[lo], pre = sP0[lo];
    for (;;) {
        const int tt = t + lane;
        const int n = tt < p.ntok ? npg_of(p, tt) : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const int before = pre + incl - n;
        const bool hit = n > 0 && (int64_t)G * before <= x && x < (int64_t)G * (before + n);
        const unsigned m = __ballot_sync(kFull, hit);
        if (m) {
            const int l = __ffs(m) - 1;
            t_out = __shfl_sync(kFull, tt, l);
            pre_out = __shfl_sync(kFull, before, l);
            return;
        }
        t += 32;
        pre += __shfl_sync(kFull, incl, 31);
    }
}

template <int kStages>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnParams p)
{
    using L = AttnSmem<kStages>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);
    const uint32_t bar_full = base + L::kBars;
    const uint32_t bar_empty = bar_full + 8 * kStages;
    const uint32_t bar_group = bar_empty + 8 * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + L::kFlag);
    volatile int* s_issued = abort_flag + 1;     // ring items the producer loaded (copies in flight at most kStages)
    volatile int* s_stop_sent = abort_flag + 2;  // the producer's final item (no data) went out
    float* sM = reinterpret_cast<float*>(sbase + L::kM);
    float* sL = reinterpret_cast<float*>(sbase + L::kL);
    int4* sMeta = reinterpret_cast<int4*>(sbase + L::kMeta);
    int* sScan = reinterpret_cast<int*>(sbase + L::kScan);
    int* sT0 = reinterpret_cast<int*>(sbase + L::kSum);
    int* sP0 = sT0 + kAttnThreads;
    int* sN = reinterpret_cast<int*>(sbase + L::kTokN);
    int* sLen = reinterpret_cast<int*>(sbase + L::kTokLen);
    int* sRow = reinterpret_cast<int*>(sbase + L::kTokRow);
    uint2* sW = reinterpret_cast<uint2*>(sbase + L::kW);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.kv_heads, H = p.heads;
    const int C = gridDim.x, c = blockIdx.x;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kConsumerWarps);
        }
        mbar_init(bar_group, kConsumerWarps);
        *abort_flag = 0;
        *s_issued = 0;
        *s_stop_sent = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    // combine_kernel may be scheduled now: its CTAs wait for this grid to finish.
    // (Every CTA of this grid is resident from the start, so they cannot block it.)
    pdl_launch_dependents();
    __syncthreads();
    // Everything below reads the call's inputs and the pool, which the kernel
    // before this one on the stream may have written.  In step mode that kernel
    // is the prompt attention, which writes nothing read here (only the prompt
    // rows of the output) and releases this grid once it has itself waited for
    // prep_kernel, whose writes this kernel reads: so this kernel starts on the
    // SMs the prompt attention leaves, and waits for it only before it exits,
    // which keeps the stream's completion order.
    if (!p.late_wait) pdl_wait();

    // ---- pages per token and their exclusive prefix over tokens (every CTA computes it).
    // The norm weights (read once here: under the kernel's own streaming a global load
    // can wait microseconds) and the first kBatch tokens' positions of each thread are
    // loaded together, one round trip.
    constexpr int kBatch = 4;
    const bool wload = !p.prepared && tid < 64;
    uint2 wv = make_uint2(0u, 0u);
    if (wload) wv = reinterpret_cast<const uint2*>(tid < 32 ? p.qw : p.kw)[tid & 31];
    const int nt = p.ntok;
    const int per = (nt + kAttnThreads - 1) / kAttnThreads;
    const int t0 = min(nt, tid * per), t1 = min(nt, t0 + per);
    int tv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) tv[k] = t0 + k < t1 ? tok_value(p, t0 + k) : 0;
    const int trow = (per == 1 && t0 < t1) ? (p.decode_mode ? t0 : p.tok_row[t0]) : 0;
    int local = 0, lmax = 0, lnz = 0;  // pages, the longest unit, tokens with pages
    auto count = [&](int n) {
        local += n;
        lmax = max(lmax, n);
        lnz += n > 0;
    };
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
        if (t0 + k < t1) count(npg_from(p, tv[k]));
    for (int t = t0 + kBatch; t < t1; ++t) count(npg_of(p, t));
    if (wload) sW[tid] = wv;
    if (per == 1) {  // every token has its own thread: what the whole-unit split reads
        sN[tid] = local;
        sLen[tid] = p.decode_mode ? tv[0] + 1 : tv[0];
        sRow[tid] = trow;
    }
    int incl = local, wmax = lmax, wnz = lnz;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
        wmax = max(wmax, __shfl_xor_sync(kFull, wmax, o));
        wnz += __shfl_xor_sync(kFull, wnz, o);
    }
    if (lane == 31) {
        sScan[warp] = incl;
        sScan[8 + warp] = wmax;
        sScan[16 + warp] = wnz;
    }
    if (p.prompt_P > 0) {
        // a step: the prompt attention's cost (prompt_tile_cost over the prompt tiles), for
        // the split of the SMs; warp w takes tiles w, w + 5, ..., kTB of them a round trip
        const int32_t* plen = p.tok_len - p.prompt_P;  // the prompt tokens' attended lengths
        const int ptiles = (p.prompt_P + 63) / 64;
        constexpr int kTB = 8, kWarps = kAttnThreads / 32;
        int64_t pc = 0;
        int pu = 0;
        for (int tb = warp; tb < ptiles; tb += kTB * kWarps) {
            int m[kTB][2];
#pragma unroll
            for (int b = 0; b < kTB; ++b)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tok = (tb + b * kWarps) * 64 + lane + 32 * i;
                    m[b][i] = (tb + b * kWarps < ptiles && tok < p.prompt_P) ? plen[tok] : 0;
                }
#pragma unroll
            for (int b = 0; b < kTB; ++b) {
                const int mx = (int)__reduce_max_sync(kFull, (uint32_t)max(max(m[b][0], m[b][1]), 0));
                pc += prompt_tile_cost(mx, G);
                pu += mx > 0 ? G : 0;
            }
        }
        if (lane == 0) {
            reinterpret_cast<int64_t*>(sbase + L::kSplit)[warp] = pc;
            reinterpret_cast<int*>(sbase + L::kSplit + 64)[warp] = pu;
        }
    }
    __syncthreads();
    int total = 0, warp_base = 0, nmax = 0, nz = 0;
#pragma unroll
    for (int w = 0; w < kAttnThreads / 32; ++w) {
        const int v = sScan[w];
        warp_base += (w < warp) ? v : 0;
        total += v;
        nmax = max(nmax, sScan[8 + w]);
        nz += sScan[16 + w];
    }
    const int excl = warp_base + incl - local;
    const int64_t T = (int64_t)G * total;
    // Ra: the CTAs resident from the start, which hold the static slices (or first units).
    // In a step the prompt attention keeps some SMs (prompt_sms), and this grid starts on
    // the others; its CTAs beyond Ra start when the prompt attention ends, and claim chunks.
    int Ra = C;
    if (p.prompt_P > 0) {
        int64_t pc = 0;
        int pu = 0;
#pragma unroll
        for (int w = 0; w < kAttnThreads / 32; ++w) {
            pc += reinterpret_cast<const int64_t*>(sbase + L::kSplit)[w];
            pu += reinterpret_cast<const int*>(sbase + L::kSplit + 64)[w];
        }
        const int pgrid = min(p.sms, ((p.prompt_P + 63) / 64) * G);  // the prompt attention's grid
        const int kept = min(prompt_sms(pc, kSplitRowPage * T, pu, p.sms), pgrid);  // the SMs it holds
        if (kept < p.sms) Ra = max(1, min(C, p.ctas_per_sm * (p.sms - kept)));
    }
    const Split sp = whole_units(nt, nmax, T, Ra) ? whole_split(G * nz, Ra) : split_of(T, Ra);
    if (sp.whole) {
        // tokens longest first (ties by index): sT0[rank] = the token, sP0[rank] = its prefix
        if (tid < nt && local > 0) {
            int rank = 0;
            for (int t = 0; t < nt; ++t) {
                const int m = sN[t];
                rank += (m > local) || (m == local && t < tid);
            }
            sT0[rank] = tid;
            sP0[rank] = excl;
        }
    } else {
        sT0[tid] = t0;
        sP0[tid] = excl;
        if (c < sp.Ce) {
            // the token holding this CTA's first page (and its prefix), found by the one
            // thread whose run of tokens holds it, so that the producer starts without a search
            const int64_t x0 = (int64_t)c * sp.S / sp.Ce;
            int run = excl;
            if (x0 >= (int64_t)G * run && x0 < (int64_t)G * (run + local)) {
                bool found = false;
                auto look = [&](int t, int n) {
                    if (!found && n > 0 && x0 < (int64_t)G * (run + n)) {
                        sScan[24] = t;
                        sScan[25] = run;
                        found = true;
                    }
                    run += n;
                };
#pragma unroll
                for (int k = 0; k < kBatch; ++k)
                    if (t0 + k < t1) look(t0 + k, npg_from(p, tv[k]));
                for (int t = t0 + kBatch; t < t1 && !found; ++t) look(t, npg_of(p, t));
            }
        }
    }
    if (c == 0) {
        int run = excl;
        for (int t = t0; t < t1; ++t) {
            p.prefix[t] = run;
            run += npg_of(p, t);
        }
        if (tid == kAttnThreads - 1) {
            p.prefix[nt] = total;
            p.prefix[nt + 1] = Ra;  // the combine derives the same intervals
        }
    }
    __syncthreads();
    if (c >= sp.Ce && !sp.ND) {  // no static slice and nothing to claim
        if (p.late_wait) pdl_wait();
        return;
    }

    if (warp == kProducerWarp) {
        // ================================================================ producer
        int i = 0;  // ring items issued
        bool ok = true;
        // Pages are read once, except the pages several rows share (a shared prompt
        // prefix): those stay in L2 for the other rows' reads, the rest go first.
        const uint64_t pol = l2_policy_evict_first(), pol_shared = l2_policy_evict_last();
        // the static slice, then one claimed chunk after another (whole-unit split:
        // unit c, then one claimed unit after another).  A chunk is claimed when
        // the range before it has kClaimAhead pages left to issue: late enough that
        // the CTAs finishing first take the chunks, early enough that the
        // counter's answer is there when the range ends.
        // (A CTA beyond the Ce static slices -- one started late, in a step -- has no
        // first range and claims at once.)
        bool stat = c < sp.Ce;  // the range is this CTA's static slice (or first unit)
        bool have = stat;       // there is a range to issue
        int64_t xb = 0, xe = 0;
        if (!sp.whole && stat) {
            xb = (int64_t)c * sp.S / sp.Ce;
            xe = (int64_t)(c + 1) * sp.S / sp.Ce;
        }
        int iv = c;     // the range's interval: partials of its pieces go to u + iv
        int unit = c;   // whole-unit split: the range's unit, in longest-first order
        uint32_t claim = 0;
        bool want = sp.ND > 0;  // the next chunk is still to be claimed
        for (;;) {
            int t = 0, pre = 0;
            if (!have) {
                xb = xe = 0;
            } else if (sp.whole) {  // one unit, never cut: no partials
                t = sT0[unit / G];
                pre = sP0[unit / G];
                const int n = sN[t];
                xb = (int64_t)G * pre + (int64_t)(unit % G) * n;
                xe = xb + n;
                iv = 0;
            } else if (stat) {  // the static slice: its first token was found in the prologue
                t = sScan[24];
                pre = sScan[25];
            } else {
                find_token(p, sT0, sP0, xb, lane, t, pre);
            }
            int64_t St = (int64_t)G * pre;  // global index of (t, kv head 0, page 0)
            int64_t x = xb;
            while (x < xe && ok) {
                const int n = sp.whole ? sN[t] : npg_of(p, t);
                const int64_t off = x - St;
                const int g = (int)(off / n), j = (int)(off % n);
                const int seg = (int)min((int64_t)(n - j), xe - x);
                int row, len;
                if (sp.whole) {
                    row = sRow[t];
                    len = sLen[t];
                } else {
                    token_info(p, t, row, len);
                }
                const int pos = len - 1;
                // lane 0: the table entry of page jj; lanes 1 and 2: the same column of the rows
                // before and after, so that a prefix page shared with a neighbouring row is known
                auto entries = [&](int jj) {
                    int e = -1;
                    if (lane < 3) {
                        const int r2 = row + (lane == 0 ? 0 : (lane == 1 ? -1 : 1));
                        if (lane == 0 || (p.table && r2 >= 0 && r2 < p.rows)) e = page_of(p.table, p.pages, r2, jj);
                    }
                    return e;
                };
                int pg_next = entries(j);  // loaded together with the row check's entries
                bool valid = true;
                if (p.decode_mode) {  // every page the row will read must be a pool page
                    int bad = 0;
                    for (int q = lane; q < n; q += 32) {
                        const int id = page_of(p.table, p.pages, row, q);
                        bad |= (id < 0 || id >= p.num_pages);
                    }
                    valid = !__any_sync(kFull, bad);
                }
                const int u = t * G + g;
                if (j == 0 && lane == 0) {  // 2: the unit is this range's alone, written out here
                    p.unit_ok[u] = valid ? (j + seg == n ? 2 : 1) : 0;
                    if (!valid && g == 0) atomicOr(p.err, PKV_DEVERR_PAGE);
                }
                const bool has_last = j + seg == n;
                const bool append = p.decode_mode && !p.prepared && valid && has_last;
                const int seg_flags = (valid ? kFlagValid : 0) | ((j == 0 && has_last) ? kFlagComplete : 0);
                for (int s = 0; s < seg; ++s, ++i) {
                    const int jj = j + s, st = i % kStages;
                    if (want && xe - (x + s) <= kClaimAhead) {
                        if (lane == 0) claim = atomicAdd(p.claim, 1u);
                        want = false;
                    }
                    if (i >= kStages &&
                        __any_sync(kFull, !mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1, p.wait_ns) ||
                                              *abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int pg = valid ? pg_next : -1;
                    if (s + 1 < seg) pg_next = entries(jj + 1);  // in flight while the next stage frees up
                    const int page = max(__shfl_sync(kFull, pg, 0), 0);
                    const int pprev = __shfl_sync(kFull, pg, 1), pnext = __shfl_sync(kFull, pg, 2);
                    const uint64_t ppol = (pprev == page || pnext == page) ? pol_shared : pol;
                    if (lane == 0) {
                        const int flags = seg_flags | (s == 0 ? kFlagFirst : 0) | (s == seg - 1 ? kFlagLast : 0) |
                                          ((s == 0 && append) ? kFlagHasLast : 0) |
                                          ((append && jj == n - 1) ? kFlagAppend : 0);
                        sMeta[2 * st] = make_int4(t, g, jj, len);
                        sMeta[2 * st + 1] = make_int4(flags, u + iv, page, 0);
                        const uint32_t fb = bar_full + 8 * st;
                        const uint32_t dst = base + st * kStageBytes;
                        uint32_t bytes = kStageBytes;
                        if (s == 0) bytes += p.prepared ? 2048 : 1536 + (append ? 1024 : 0);
                        mbar_arrive_expect_tx(fb, bytes);
                        const int y = page * kPageSize;
                        tma_load_3d(dst, &tmK, 0, y, g, fb, ppol);
                        tma_load_3d(dst + 8192, &tmK, 64, y, g, fb, ppol);
                        tma_load_3d(dst + 16384, &tmV, 0, y, g, fb, ppol);
                        tma_load_3d(dst + 24576, &tmV, 64, y, g, fb, ppol);
                        if (s == 0 && p.prepared) {  // the 4 heads' prepared q, fp32
                            const uint32_t side = base + L::kSide + st * kSideBytes;
                            bulk_copy(side, p.qhat + ((int64_t)t * H + g * kGroup) * kHeadDim, 2048, fb);
                        } else if (s == 0) {
                            const uint32_t side = base + L::kSide + st * kSideBytes;
                            bulk_copy(side + kSideQ, p.q + ((int64_t)t * H + g * kGroup) * kHeadDim, 1024, fb);
                            bulk_copy(side + kSideRopeHi, p.rope_hi + (int64_t)pos * kRopeHalf, 512, fb);
                            if (append) {
                                const int64_t kv = ((int64_t)t * G + g) * kHeadDim;
                                bulk_copy(side + kSideRopeLo, p.rope_lo + (int64_t)pos * kRopeHalf, 512, fb);
                                bulk_copy(side + kSideK, p.k + kv, 256, fb);
                                bulk_copy(side + kSideV, p.v + kv, 256, fb);
                            }
                        }
                    }
                    __syncwarp();
                }
                x += seg;
                if (ok && x < xe && x >= St + (int64_t)G * n) {  // next token that has pages
                    St += (int64_t)G * n;
                    do {
                        ++t;
                    } while (npg_of(p, t) == 0);
                }
            }
            if (!ok || !sp.ND) break;
            if (want && lane == 0) claim = atomicAdd(p.claim, 1u);  // (a range that issued nothing)
            want = true;
            const uint32_t k = __shfl_sync(kFull, claim, 0);
            if (k >= (uint32_t)sp.ND) break;
            stat = false;
            have = true;
            unit = sp.Ce + (int)k;
            xb = sp.S + (int64_t)k * sp.Q;
            xe = xb + sp.Q;
            iv = sp.Ce + (int)k;
        }
        if (ok) {  // the end: a ring item without data that stops the consumers
            const int st = i % kStages;
            if (i >= kStages &&
                __any_sync(kFull, !mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1, p.wait_ns) || *abort_flag)) {
                ok = false;
            } else if (lane == 0) {
                sMeta[2 * st + 1] = make_int4(kFlagStop, 0, 0, 0);
                mbar_arrive(bar_full + 8 * st);
                *s_stop_sent = 1;
            }
            __syncwarp();
        }
        if (lane == 0) {
            *s_issued = i;
            if (!ok) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {

        // ==================================================================== consumers
        const int gid = lane >> 2, tig = lane & 3;
        // This lane's B fragments hold dims 16ks + 2tig + {0, 1, 8, 9} (ks = 0..7) of
        // one query head: 32 dims, closed under the rotate-half pairing (d, d +- 64),
        // and the four lanes tig = 0..3 of a head hold all 128 of its dims.
        const uint32_t* sWq = reinterpret_cast<const uint32_t*>(sW);  // q_norm_w as bf16 pairs
        uint32_t wq2[8][2];  // q_norm weights of those dims, bf16 pairs
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int d0 = 16 * ks + 2 * tig;
            wq2[ks][0] = sWq[d0 >> 1];
            wq2[ks][1] = sWq[(d0 + 8) >> 1];
        }
        float wk[4];
        unpack4(sW[32 + lane], wk);
        const float qscale = 1.4426950408889634f * 0.088388347648318440f;  // log2(e) / sqrt(128)
        const bool rem_lane = tig >= 2;  // this lane's S/O columns are the remainder columns
        const int hh = gid & 3, prt = gid >> 2;
        const int srcA = 4 * (2 * tig) + (hh >> 1) + 2 * prt;  // lanes holding P for the PV B fragment
        const int srcB = srcA + 4;
        const int r_ld = lane & 7, j_ld = lane >> 3;
        uint32_t gphase = 0;

        uint32_t bq[8][2];
        float o[8][4];
        float mA = -CUDART_INF_F, mB = -CUDART_INF_F, lA = 0.f, lB = 0.f;
        uint2 knew = make_uint2(0u, 0u), vnew = make_uint2(0u, 0u);  // the row's new k (normed, roped) and v
        bool ok = true;

        for (int i = 0;; ++i) {
            const int st = i % kStages;
            if (__any_sync(kFull, !mbar_wait(bar_full + 8 * st, (i / kStages) & 1, p.wait_ns))) {
                ok = false;
                break;
            }
            const int4 m1 = sMeta[2 * st + 1];
            const int flags = m1.x;
            if (flags & kFlagStop) break;
            const int4 m0 = sMeta[2 * st];
            const int t = m0.x, g = m0.y, jj = m0.z, len = m0.w, pidx = m1.y, page = m1.z;
            const uint32_t kb = base + st * kStageBytes;
            const uint32_t vb = kb + 16384;

            if ((flags & kFlagFirst) && p.prepared) {
                q_from_hat(reinterpret_cast<const float*>(sbase + L::kSide + st * kSideBytes) + hh * kHeadDim, qscale,
                           tig, prt, bq);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
                mA = mB = -CUDART_INF_F;
                lA = lB = 0.f;
            } else if (flags & kFlagFirst) {
                const uint8_t* side = sbase + L::kSide + st * kSideBytes;
                const float2* rpf = reinterpret_cast<const float2*>(side + kSideRopeHi);
                // q of head 4g+hh, the dims of this lane's B fragments: QK-norm + RoPE in
                // fp32 from the raw q and (cos, sin) staged with this page, scaled by
                // log2(e)/sqrt(128), then split into bf16 head (cols 0-3) and remainder (cols 4-7)
                {
                    const uint8_t* qrow = side + hh * 256;
                    uint32_t xr[8][2];
                    float ss = 0.f;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int d0 = 16 * ks + 2 * tig;
                        xr[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 2 * d0);
                        xr[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 2 * (d0 + 8));
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float a = __uint_as_float(xr[ks][e] << 16), b = __uint_as_float(xr[ks][e] & 0xffff0000u);
                            ss += a * a + b * b;
                        }
                    }
                    ss += __shfl_xor_sync(kFull, ss, 1);
                    ss += __shfl_xor_sync(kFull, ss, 2);
                    const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps) * qscale;
                    switch (p.rot) {  // rotated dims: pairs (d, d + rot / 2)
                    case 128: q_prep<4>(xr, wq2, rpf, inv, tig, prt, bq); break;
                    case 96: q_prep<3>(xr, wq2, rpf, inv, tig, prt, bq); break;
                    case 64: q_prep<2>(xr, wq2, rpf, inv, tig, prt, bq); break;
                    default: q_prep<1>(xr, wq2, rpf, inv, tig, prt, bq); break;
                    }
                }
                // the warp that owns the new slot's position prepares the row's k and v
                if ((flags & kFlagHasLast) && warp == ((len - 1) % kPageSize) / 16) {
                    knew = norm_rope_k(*reinterpret_cast<const uint2*>(side + kSideK + 8 * lane), wk, rpf,
                                       reinterpret_cast<const float2*>(side + kSideRopeLo), p.eps, lane, p.rot);
                    vnew = *reinterpret_cast<const uint2*>(side + kSideV + 8 * lane);
                }
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
                mA = mB = -CUDART_INF_F;
                lA = lB = 0.f;
            }

            if ((flags & kFlagAppend) && warp == ((len - 1) % kPageSize) / 16) {
                // the page holding the row's new slot: write k and v into the staged
                // page (row r of the 128-byte-swizzled halves) and into the pool
                const int r = (len - 1) % kPageSize;
                const int half = lane >> 4, chunk = (lane & 15) >> 1;
                const uint32_t off = half * 8192 + r * 128 + ((chunk ^ (r & 7)) << 4) + (lane & 1) * 8;
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(kb + off), "r"(knew.x), "r"(knew.y) : "memory");
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(vb + off), "r"(vnew.x), "r"(vnew.y) : "memory");
                const int64_t slot = (int64_t)page * kPageSize + r;
                const int64_t dst = ((int64_t)g * p.num_slots + slot) * kHeadDim + 4 * lane;
                *reinterpret_cast<uint2*>(p.K + dst) = knew;
                *reinterpret_cast<uint2*>(p.V + dst) = vnew;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before TMA refills this stage
                __syncwarp();
            }

            // ---- S = K q^T (two accumulators for ILP)
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const int rowk = 16 * warp + r_ld + 8 * (j_ld & 1);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int cc = 2 * ks + (j_ld >> 1);
                    const uint32_t addr = kb + (ks >> 2) * 8192 + rowk * 128 + (((cc & 7) ^ (rowk & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(addr, a0, a1, a2, a3);
                    if (ks & 1)
                        mma_bf16_16816(c1, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
                    else
                        mma_bf16_16816(c0, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
                }
            }
            float sv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sv[k] = c0[k] + c1[k];
                sv[k] += __shfl_xor_sync(kFull, sv[k], 2);  // head column + remainder column
            }
            // sv[0]: (pos gid, head A), sv[1]: (gid, B), sv[2]: (gid+8, A), sv[3]: (gid+8, B)
            const int pbase = jj * kPageSize + 16 * warp;
            if (pbase + gid >= len) sv[0] = sv[1] = -CUDART_INF_F;
            if (pbase + gid + 8 >= len) sv[2] = sv[3] = -CUDART_INF_F;

            float tA = fmaxf(sv[0], sv[2]), tB = fmaxf(sv[1], sv[3]);
#pragma unroll
            for (int o2 = 4; o2 < 32; o2 <<= 1) {
                tA = fmaxf(tA, __shfl_xor_sync(kFull, tA, o2));
                tB = fmaxf(tB, __shfl_xor_sync(kFull, tB, o2));
            }
            const float nA = fmaxf(mA, tA), nB = fmaxf(mB, tB);
            const float aA = (nA == -CUDART_INF_F) ? 1.f : exp2f(mA - nA);
            const float aB = (nB == -CUDART_INF_F) ? 1.f : exp2f(mB - nB);
            float pv[4];
            pv[0] = (sv[0] == -CUDART_INF_F) ? 0.f : exp2f(sv[0] - nA);
            pv[1] = (sv[1] == -CUDART_INF_F) ? 0.f : exp2f(sv[1] - nB);
            pv[2] = (sv[2] == -CUDART_INF_F) ? 0.f : exp2f(sv[2] - nA);
            pv[3] = (sv[3] == -CUDART_INF_F) ? 0.f : exp2f(sv[3] - nB);
            lA = lA * aA + pv[0] + pv[2];
            lB = lB * aB + pv[1] + pv[3];
            mA = nA;
            mB = nB;
            if (aA != 1.f || aB != 1.f) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    o[mt][0] *= aA;
                    o[mt][1] *= aB;
                    o[mt][2] *= aA;
                    o[mt][3] *= aB;
                }
            }

            // ---- P fragment: this lane provides head-or-remainder parts of its four p values
            uint32_t w_even, w_odd;
            {
                __nv_bfloat16 e[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    __nv_bfloat16 hd, tl;
                    split_bf16(pv[k], hd, tl);
                    e[k] = rem_lane ? tl : hd;
                }
                w_even = pack_bf16(e[0], e[2]);  // head A at positions gid, gid+8
                w_odd = pack_bf16(e[1], e[3]);   // head B
            }
            const uint32_t xae = __shfl_sync(kFull, w_even, srcA), xao = __shfl_sync(kFull, w_odd, srcA);
            const uint32_t xbe = __shfl_sync(kFull, w_even, srcB), xbo = __shfl_sync(kFull, w_odd, srcB);
            const uint32_t XA = (hh & 1) ? xao : xae;  // {P[2tig][col], P[2tig+8][col]}
            const uint32_t XB = (hh & 1) ? xbo : xbe;  // {P[2tig+1][col], P[2tig+9][col]}
            const uint32_t pb0 = __byte_perm(XA, XB, 0x5410);
            const uint32_t pb1 = __byte_perm(XA, XB, 0x7632);

            // ---- O^T += V^T P
            {
                const int rowv = 16 * warp + r_ld + 8 * (j_ld >> 1);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int cc = 2 * mt + (j_ld & 1);
                    const uint32_t addr = vb + (mt >> 2) * 8192 + rowv * 128 + (((cc & 7) ^ (rowv & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4_trans(addr, a0, a1, a2, a3);
                    mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
                }
            }
            __syncwarp();
            if (!(flags & kFlagLast)) {
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            } else {
                // ---- end of segment: merge the four warps in a fixed order, write the output or a partial.
                // Each warp parks its unscaled O in the K rows of this stage that only it read
                // (rows 16w..16w+15 of the first half: 2 KiB), its m and l in sM/sL.
                float lAs = lA, lBs = lB;
#pragma unroll
                for (int o2 = 4; o2 < 32; o2 <<= 1) {
                    lAs += __shfl_xor_sync(kFull, lAs, o2);
                    lBs += __shfl_xor_sync(kFull, lBs, o2);
                }
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                    for (int k = 0; k < 4; ++k) o[mt][k] += __shfl_xor_sync(kFull, o[mt][k], 2);
                float* park = reinterpret_cast<float*>(sbase + st * kStageBytes);  // [4 warps][4 heads][128]
                if (tig < 2) {
                    const int hA = 2 * tig, hB = hA + 1;
                    float* pa = park + (warp * 4 + hA) * kHeadDim;
                    float* pb = park + (warp * 4 + hB) * kHeadDim;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int d = 16 * mt + gid;
                        pa[d] = o[mt][0];
                        pb[d] = o[mt][1];
                        pa[d + 8] = o[mt][2];
                        pb[d + 8] = o[mt][3];
                    }
                    if (gid == 0) {
                        sM[warp * 4 + hA] = mA;
                        sM[warp * 4 + hB] = mB;
                        sL[warp * 4 + hA] = lAs;
                        sL[warp * 4 + hB] = lBs;
                    }
                }
                if (!group_sync(bar_group, gphase, lane, p.wait_ns)) {
                    ok = false;
                    break;
                }
                {
                    const int h = warp;  // thread -> (head h, dims 4*lane..4*lane+3)
                    float M = -CUDART_INF_F;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sM[w * 4 + h]);
                    float Ls = 0.f, y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {  // fixed order: the result is reproducible
                        const float mw = sM[w * 4 + h];
                        const float f = (mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
                        Ls += f * sL[w * 4 + h];
                        const float4 ow = *reinterpret_cast<const float4*>(park + (w * 4 + h) * kHeadDim + 4 * lane);
                        y[0] += f * ow.x;
                        y[1] += f * ow.y;
                        y[2] += f * ow.z;
                        y[3] += f * ow.w;
                    }
                    const float inv = 1.f / Ls;
#pragma unroll
                    for (int k = 0; k < 4; ++k) y[k] *= inv;
                    const int qh = g * kGroup + h;
                    if (flags & kFlagComplete) {
                        if (!(flags & kFlagValid)) y[0] = y[1] = y[2] = y[3] = 0.f;
                        *reinterpret_cast<uint2*>(p.out + ((int64_t)t * H + qh) * kHeadDim + 4 * lane) = pack4(y);
                    } else {
                        const int64_t ph = (int64_t)pidx * kGroup + h;
                        *reinterpret_cast<float4*>(p.part_o + ph * kHeadDim + 4 * lane) =
                            make_float4(y[0], y[1], y[2], y[3]);
                        if (lane == 0) p.part_lse[ph] = M + log2f(Ls);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before TMA refills this stage
                if (!group_sync(bar_group, gphase, lane, p.wait_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            }
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }
    // Every role has stopped.  After an abort, copies of up to kStages ring items
    // may still be landing in this CTA's shared memory: wait for them (with the
    // full limit, whatever the call's wait limit) before the CTA exits.
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        const int n = *s_issued;
        // the stop item, when sent, reused the stage of item n - kStages, which had landed
        for (int k2 = max(0, n - kStages + (*s_stop_sent ? 1 : 0)); k2 < n; ++k2)
            mbar_wait(bar_full + 8 * (k2 % kStages), (k2 / kStages) & 1, kWaitLimitNs);
    }
    if (p.late_wait) pdl_wait();
}

constexpr int kAttnStages = 3;

int attn_ctas_per_sm()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<kAttnStages>, kAttnThreads,
                                                      AttnSmem<kAttnStages>::kAlloc) != cudaSuccess)
        return 0;
    return n;
}

cudaError_t configure_kernels()
{
    return cudaFuncSetAttribute(attn_kernel<kAttnStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnSmem<kAttnStages>::kAlloc);
}

cudaError_t launch_attn(const pkv_pool* pool, const StepArgs& a, const Plan& plan, bool decode_mode, bool pdl,
                        cudaStream_t s)
{
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.k = static_cast<const __nv_bfloat16*>(a.k);
    p.v = static_cast<const __nv_bfloat16*>(a.v);
    p.qw = static_cast<const __nv_bfloat16*>(a.q_norm_w);
    p.kw = static_cast<const __nv_bfloat16*>(a.k_norm_w);
    p.positions = a.step_positions;
    p.tok_len = reinterpret_cast<const int32_t*>(a.ws + plan.off_len);
    p.tok_row = reinterpret_cast<const int32_t*>(a.ws + plan.off_row);
    p.table = a.table;
    p.rope_hi = pool->rope_hi;
    p.rope_lo = pool->rope_lo;
    p.K = static_cast<__nv_bfloat16*>(pool->k);
    p.V = static_cast<__nv_bfloat16*>(pool->v);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.part_o = reinterpret_cast<float*>(a.ws + plan.off_po);
    p.part_lse = reinterpret_cast<float*>(a.ws + plan.off_plse);
    p.claim = plan.claim;
    p.prefix = reinterpret_cast<int32_t*>(a.ws + plan.off_prefix);
    p.unit_ok = reinterpret_cast<int32_t*>(a.ws + plan.off_unit_ok);
    p.err = pool->err;
    p.ntok = plan.tokens;
    p.pages = a.pages;
    p.rows = a.rows;
    p.num_pages = pool->num_pages;
    p.max_seq = pool->cfg.max_seq;
    p.heads = pool->cfg.heads;
    p.kv_heads = pool->cfg.kv_heads;
    p.decode_mode = decode_mode ? 1 : 0;
    p.qhat = a.q_hat;
    p.prepared = a.q_hat ? 1 : 0;
    p.late_wait = (!decode_mode && pdl) ? 1 : 0;
    // a step whose prompt attention runs beside this kernel (programmatic launch) splits the SMs
    p.prompt_P = p.late_wait ? a.P : 0;
    p.sms = pool->num_sms;
    p.ctas_per_sm = pool->ctas_per_sm;
    p.rot = pool->cfg.rotary_dim > 0 ? pool->cfg.rotary_dim : kHeadDim;
    p.num_slots = pool->num_slots;
    p.eps = static_cast<float>(pool->cfg.eps);
    p.wait_ns = pool->wait_ns;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.ctas);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = AttnSmem<kAttnStages>::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_kernel<kAttnStages>, pool->tmap_k, pool->tmap_v, p);
}

// =====================================================================================
// combine_kernel
// =====================================================================================
struct CombineParams {
    const int32_t* prefix;    // [ntok + 2]: page prefix, total, the attention's resident CTAs
    const int32_t* unit_ok;   // [U]
    const int32_t* positions; // decode mode: [ntok]
    const float* part_o;
    const float* part_lse;
    __nv_bfloat16* out;
    uint32_t* err;
    uint32_t* claim;          // the attention's chunk counter: zeroed here for the call that next uses it
    int ntok, heads, kv_heads, decode_mode;
};

// One CTA per (token, kv head) unit; warp w = query head 4g+w, lane owns dims 4*lane..4*lane+3.
//   out = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M)   over the unit's pieces c
template <int kBatch, int kWph>
__global__ void __launch_bounds__(128 * kWph) combine_kernel(CombineParams p)
{
    // warp w merges query head w % 4 of the unit's kv group; with kWph warps a
    // head, warp w takes every kWph-th piece from piece w / 4 on
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hw = warp % kGroup, sub = warp / kGroup;
    const int G = p.kv_heads;
    const int u = blockIdx.x;
    const int t = u / G, g = u % G;
    const int h = g * kGroup + hw;
    pdl_wait();
    if (u == 0 && threadIdx.x == 0) *p.claim = 0;  // the attention grid has finished claiming
    __nv_bfloat16* dst = p.out + ((int64_t)t * p.heads + h) * kHeadDim + 4 * lane;
    // every index this CTA needs, loaded together (one round trip)
    const int pre = p.prefix[t], pre1 = p.prefix[t + 1], total = p.prefix[p.ntok], ra = p.prefix[p.ntok + 1];
    const int uok = p.unit_ok[u];
    const int n = pre1 - pre;
    if (n == 0) {  // skipped token
        if (sub == 0) *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
        if (p.decode_mode && g == 0 && threadIdx.x == 0) {
            const int pos = p.positions[t];
            if (pos != -1) atomicOr(p.err, PKV_DEVERR_POSITION);
        }
        return;
    }
    if (!uok) {
        if (sub == 0) *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
        return;
    }
    if (uok == 2) return;  // one range held the whole unit, and its CTA wrote it out
    const int64_t T = (int64_t)G * total;
    const Split sp = split_of(T, ra);  // the attention kernel's intervals (ra: its static slices' CTAs)
    const int64_t S = (int64_t)G * pre + (int64_t)g * n;
    const int64_t rf = interval_of(S, sp), rl = interval_of(S + n - 1, sp);
    if (rf == rl) return;  // one interval held the whole unit, and its CTA wrote it out
    // the pieces' log-sum-exps, one per lane, and this warp's first kPre pieces'
    // partial outputs, all in flight together (a second round trip); then the
    // rest of this warp's pieces in order, in batches of kBatch whose loads are
    // all issued before the first is summed (a unit split over many chunks, as a
    // few long rows are, would otherwise pay a round trip every few pieces)
    constexpr int kPre = 4;
    static_assert(kPre * kWph <= 32 && 32 % kWph == 0, "the first pieces lie in the first block of 32");
    const int np = (int)(rl - rf + 1);
    const float* lse = p.part_lse + ((int64_t)u + rf) * kGroup + hw;
    const float* po = p.part_o + (((int64_t)u + rf) * kGroup + hw) * kHeadDim + 4 * lane;
    const int64_t ostride = (int64_t)kGroup * kHeadDim;
    const float l0 = lane < np ? lse[(int64_t)lane * kGroup] : -CUDART_INF_F;
    float4 ob[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int r = sub + k * kWph;
        ob[k] = r < np ? *reinterpret_cast<const float4*>(po + r * ostride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float M = l0;
    for (int r = lane + 32; r < np; r += 32) M = fmaxf(M, lse[(int64_t)r * kGroup]);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o2));
    const float wl0 = lane < np ? exp2f(l0 - M) : 0.f;
    float wsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kPre; ++k) {  // pieces beyond np add w = 0 times o = 0
        const float w = __shfl_sync(kFull, wl0, sub + k * kWph);
        wsum += w;
        acc[0] += w * ob[k].x;
        acc[1] += w * ob[k].y;
        acc[2] += w * ob[k].z;
        acc[3] += w * ob[k].w;
    }
    for (int r0 = 0; r0 < np; r0 += 32) {
        const int nb = min(32, np - r0);
        const float wl = r0 == 0 ? wl0 : (lane < nb ? exp2f(lse[(int64_t)(r0 + lane) * kGroup] - M) : 0.f);
        for (int r = r0 == 0 ? sub + kPre * kWph : sub; r < nb; r += kWph * kBatch) {
            float4 o[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (r + i * kWph < nb) o[i] = *reinterpret_cast<const float4*>(po + (r0 + r + i * kWph) * ostride);
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (r + i * kWph >= nb) break;  // the same on every lane
                const float w = __shfl_sync(kFull, wl, r + i * kWph);
                wsum += w;
                acc[0] += w * o[i].x;
                acc[1] += w * o[i].y;
                acc[2] += w * o[i].z;
                acc[3] += w * o[i].w;
            }
        }
    }
    if constexpr (kWph > 1) {  // the head's warps' sums, added in warp order
        __shared__ float part[kWph][kGroup][32][5];
        float* mine = part[sub][hw][lane];
        mine[0] = acc[0], mine[1] = acc[1], mine[2] = acc[2], mine[3] = acc[3], mine[4] = wsum;
        __syncthreads();
        if (sub != 0) return;
#pragma unroll
        for (int q = 1; q < kWph; ++q) {
            const float* o = part[q][hw][lane];
            acc[0] += o[0], acc[1] += o[1], acc[2] += o[2], acc[3] += o[3], wsum += o[4];
        }
    }
    const float inv = 1.f / wsum;
    const float y[4] = {acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv};
    *reinterpret_cast<uint2*>(dst) = pack4(y);
}

cudaError_t launch_combine(const pkv_pool* pool, const StepArgs& a, const Plan& plan, bool decode_mode,
                           cudaStream_t s)
{
    CombineParams p;
    p.prefix = reinterpret_cast<const int32_t*>(a.ws + plan.off_prefix);
    p.unit_ok = reinterpret_cast<const int32_t*>(a.ws + plan.off_unit_ok);
    p.positions = a.step_positions;
    p.part_o = reinterpret_cast<const float*>(a.ws + plan.off_po);
    p.part_lse = reinterpret_cast<const float*>(a.ws + plan.off_plse);
    p.claim = plan.claim;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.err = pool->err;
    p.ntok = plan.tokens;
    p.heads = pool->cfg.heads;
    p.kv_heads = pool->cfg.kv_heads;
    p.decode_mode = decode_mode ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)plan.tokens * pool->cfg.kv_heads));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Few units for the grid (a few long rows): each is split over many chunks, and the
    // combine's CTAs are few, so each loads 16 pieces at a time, and under half a unit a
    // CTA, four warps share each query head.  Otherwise 8 at a time keep the kernel at 64
    // registers, two of its CTAs resident beside the attention's.
    const int64_t units = (int64_t)plan.tokens * pool->cfg.kv_heads;
    if (2 * units < (int64_t)plan.ctas) {
        cfg.blockDim = dim3(128 * 4);
        return cudaLaunchKernelEx(&cfg, combine_kernel<16, 4>, p);
    }
    if (units < 2 * (int64_t)plan.ctas) return cudaLaunchKernelEx(&cfg, combine_kernel<16, 1>, p);
    return cudaLaunchKernelEx(&cfg, combine_kernel<8, 1>, p);
}

// =====================================================================================
// output gate of the gated-attention variant: out *= sigmoid(gate), elementwise
// (fantasma model.zig, fullAttentionForward: "attn_out *= sigmoid(gate)")
// =====================================================================================
__global__ void __launch_bounds__(256) gate_kernel(__nv_bfloat16* out, const __nv_bfloat16* gate, int64_t n8)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 o = reinterpret_cast<const uint4*>(out)[i], g = reinterpret_cast<const uint4*>(gate)[i];
        const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
        uint32_t r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float y[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const float x = __uint_as_float(b ? (ov[e] & 0xffff0000u) : (ov[e] << 16));
                const float z = __uint_as_float(b ? (gv[e] & 0xffff0000u) : (gv[e] << 16));
                y[b] = x / (1.f + expf(-z));
            }
            const __nv_bfloat162 t = __floats2bfloat162_rn(y[0], y[1]);
            r[e] = *reinterpret_cast<const uint32_t*>(&t);
        }
        reinterpret_cast<uint4*>(out)[i] = make_uint4(r[0], r[1], r[2], r[3]);
    }
}

cudaError_t launch_gate(const pkv_pool* pool, void* out, const void* gate, int64_t n, cudaStream_t s)
{
    const int64_t n8 = n / 8;
    const int64_t want = (n8 + 255) / 256, cap = 8LL * pool->num_sms;
    gate_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, s>>>(static_cast<__nv_bfloat16*>(out),
                                                                    static_cast<const __nv_bfloat16*>(gate), n8);
    return cudaGetLastError();
}

}  // namespace pkv
