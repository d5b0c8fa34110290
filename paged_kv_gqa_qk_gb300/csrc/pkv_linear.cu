// The projections either side of the attention: y = x W^T on tcgen05 tensor
// cores (sm_103a).
//
// qwen3-8b Nest files, src/attention.linnet, GroupedQueryAttention.decode_paged
// and step_paged: q_proj, k_proj and v_proj map the layer input x [tokens][4096]
// to q [tokens][32 x 128] and k, v [tokens][8 x 128] before split_heads; o_proj
// maps merge_heads of the attention output back to [tokens][4096].  Each is a
// linear map without bias (README.md: "The query and key projections carry no
// bias"), y[t][o] = sum_k x[t][k] w[o][k] with w in nn.Linear layout [out][in].
//
// A CTA computes a tile of 128 output features x BN tokens, D = W_tile x_tile^T
// with M = 128 (rows of W), N = BN (tokens), accumulated over the input
// features in steps of 64 in tensor memory (lane = output feature, column =
// token).  Warp 0 streams the W and x boxes through a ring with TMA, warp 1
// allocates tensor memory and one of its threads issues the MMAs, and all four
// warps read the accumulator back and write y (lanes of a warp write 32
// consecutive output features of one token: 64 contiguous bytes).  When the
// tiles alone would leave most SMs idle (few tokens: the decode step), the
// input features are split over the `splits` CTAs of a thread-block cluster:
// each stages its fp32 partial tile in its own shared memory, and CTA r of the
// cluster sums slice r of the features over all of them (distributed shared
// memory, in a fixed order) and writes it.
#include <cuda_bf16.h>

#include <type_traits>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "pkv_rope.cuh"

namespace pkv {

namespace {

constexpr int kLinThreads = 128;
constexpr int kBM = 128;         // output features per tile (M)
constexpr int kBK = 64;          // input features per ring stage (one 128-byte swizzle span)
constexpr int kMaxSplits = 8;    // a portable cluster

template <int BN>
struct LinShape {
    static constexpr int kABytes = kBM * kBK * 2;  // 16 KiB of W
    static constexpr int kBBytes = BN * kBK * 2;   // x
    static constexpr int kStageBytes = kABytes + kBBytes;
    // 64-token tiles (the decode step) keep two CTAs per SM resident: 96 KiB rings
    static constexpr int kStages = BN == 64 ? 4 : (192 * 1024) / kStageBytes;
    static_assert(kStages * kStageBytes >= kBM * BN * 4, "the ring holds the fp32 partial tile");
    static constexpr int kBars = kStages * kStageBytes;  // full[S], empty[S], done
    static constexpr int kTmemSlot = kBars + 8 * (2 * kStages + 1);
    static constexpr int kTok = (kTmemSlot + 16 + 15) / 16 * 16;  // fused epilogue: int2 (position, slot) per token
    static constexpr int kAlloc = kTok + 8 * BN + 1024;
};

// The q/k/v projection with the per-token work before attention fused into
// its epilogue (pkv_qkv_proj_append): each 128-feature tile is one head, so the
// CTA that finishes a token's head of q, k or v holds all of it.  Token t is a
// decode row (table row t) at positions[t]; qhat receives its QK-normed, roped
// q in fp32, and its normed, roped k (bf16) and its v go straight to its slot
// of the pool.  Rows the attention skips (position -1, or a position or page
// it cannot read) are not written.
struct LinFuse {
    const __nv_bfloat16* qw;   // q_norm weights [128]
    const __nv_bfloat16* kw;   // k_norm weights [128]
    const int32_t* positions;  // [tokens]
    const int32_t* table;      // [tokens][pages], or null: contiguous rows
    const float2* rope_hi;     // (cos, sin) [max_seq][64]
    const float2* rope_lo;
    __nv_bfloat16* K;          // pool [kv_heads][num_slots][128]
    __nv_bfloat16* V;
    float* qhat;               // [tokens][heads][128]
    int64_t num_slots;
    int pages, num_pages, max_seq, rot, heads;
    float eps;
};

// The output features split into up to three consecutive segments, each
// written to its own [tokens][width] tensor (q, k, v of one fused projection);
// segment boundaries are multiples of 128, so a tile lies in one segment.
struct LinParams {
    __nv_bfloat16* y[3];
    int seg_end[3];     // cumulative widths; seg_end[2] == out
    uint32_t* err;
    int tokens, in, out, splits;
    int fused;          // 1: the epilogue of LinFuse instead of writing y
    LinFuse f;
};

// The tokens of the tile this CTA finishes in the fused epilogue: all BN
// without a split, tokens [r BN / NS, (r + 1) BN / NS) for CTA r of a cluster of NS.
__device__ __forceinline__ void fused_token_range(const LinParams& p, int bn, int& t_lo, int& t_hi)
{
    const int ns = p.splits, r = ns > 1 ? (int)cluster_rank() : 0;
    t_lo = r * bn / ns;
    t_hi = (r + 1) * bn / ns;
}

// Run by warps 2 and 3 while the product runs: for each token t of the range,
// tok[t - t_lo] = (position, slot), or position -1 for a token nothing is
// written for -- no step (-1), a position out of range or a page the attention
// cannot read (these set the error bits, from the CTAs of k's first head) --
// and for rows past the batch.
__device__ __forceinline__ void fused_tokens(const LinParams& p, int2* tok, int bn, int n0, int m0, int w2, int lane)
{
    const LinFuse& f = p.f;
    int t_lo, t_hi;
    fused_token_range(p, bn, t_lo, t_hi);
    const bool reporter = m0 == p.seg_end[0];  // the tile of k's head 0
    for (int t = t_lo + w2; t < t_hi; t += 2) {
        const int tk = n0 + t;
        int pos = tk < p.tokens ? f.positions[tk] : -1;
        uint32_t e = 0;
        if (pos != -1 && (pos < 0 || pos >= f.max_seq || pos >= f.pages * kPageSize)) e = PKV_DEVERR_POSITION;
        int bad = 0;
        if (pos >= 0 && !e)
            for (int j = lane; j <= pos / kPageSize; j += 32) {
                const int id = page_of(f.table, f.pages, tk, j);
                bad |= (id < 0 || id >= f.num_pages);
            }
        if (__any_sync(kFull, bad)) e = PKV_DEVERR_PAGE;
        int slot = 0;
        if (e || pos < 0)
            pos = -1;
        else
            slot = page_of(f.table, f.pages, tk, pos / kPageSize) * kPageSize + pos % kPageSize;
        if (lane == 0) {
            tok[t - t_lo] = make_int2(pos, slot);
            if (e && reporter) atomicOr(p.err, e);
        }
    }
}

// Fused epilogue for this CTA's tokens of the tile (rows n0 + t): warp w takes
// the range's tokens w, w + 4, ...; lane l sums features 4l..4l+3 of the token
// over the NS partial tiles [token][feature] fp32 at the cluster addresses src
// (NS = 1: this CTA's own tile, plain shared memory), rounds them to bf16 --
// the projection's output, as the pages' q/k/v tensors are bf16 -- and does
// the segment's work: q -> norm + rope -> qhat; k -> norm + rope -> K[slot];
// v -> V[slot].  The (position, slot) of each token come from fused_tokens; a
// warp takes two tokens a pass and has all their loads in flight at once.
template <int NS>
__device__ __forceinline__ void fused_rows(const LinParams& p, const uint32_t (&src)[NS], const float* own,
                                           const int2* tok, int bn, int n0, int m0, int warp, int lane)
{
    const LinFuse& f = p.f;
    const int seg = m0 < p.seg_end[0] ? 0 : (m0 < p.seg_end[1] ? 1 : 2);
    const int head = (m0 - (seg ? p.seg_end[seg - 1] : 0)) / kBM;
    const KRope kr = krope(lane, f.rot);
    float w4[4] = {0.f, 0.f, 0.f, 0.f};
    if (seg < 2) unpack4(reinterpret_cast<const uint2*>(seg == 0 ? f.qw : f.kw)[lane], w4);
    int t_lo, t_hi;
    fused_token_range(p, bn, t_lo, t_hi);
    // (cos, sin) hi (and lo, for k) of this lane's table entries at a token's position
    auto rope_rows = [&](int pos, float2 (&rh)[4], float2 (&rl)[4]) {
        if (pos < 0 || seg == 2) return;
        const float4* h4 = reinterpret_cast<const float4*>(f.rope_hi + (int64_t)pos * kRopeHalf + kr.f0);
        const float4 h0 = h4[0], h1 = h4[1];
        rh[0] = make_float2(h0.x, h0.y), rh[1] = make_float2(h0.z, h0.w), rh[2] = make_float2(h1.x, h1.y),
        rh[3] = make_float2(h1.z, h1.w);
        if (seg == 1) {
            const float4* l4 = reinterpret_cast<const float4*>(f.rope_lo + (int64_t)pos * kRopeHalf + kr.f0);
            const float4 l0 = l4[0], l1 = l4[1];
            rl[0] = make_float2(l0.x, l0.y), rl[1] = make_float2(l0.z, l0.w), rl[2] = make_float2(l1.x, l1.y),
            rl[3] = make_float2(l1.z, l1.w);
        }
    };
    // the projected values of token t (features 4l..4l+3), summed over the NS partial tiles
    auto partial = [&](int t, float4 (&v)[NS]) {
        if (NS == 1) {
            v[0] = reinterpret_cast<const float4*>(own)[t * (kBM / 4) + lane];
        } else {
#pragma unroll
            for (int q = 0; q < NS; ++q) v[q] = ld_cluster_f32x4(src[q] + (uint32_t)(t * kBM + 4 * lane) * 4);
        }
    };
    auto finish = [&](int t, const int2 cur, const float4 (&v)[NS], const float2 (&rh)[4], const float2 (&rl)[4]) {
        float4 a = v[0];
#pragma unroll
        for (int q = 1; q < NS; ++q) {
            a.x += v[q].x;
            a.y += v[q].y;
            a.z += v[q].z;
            a.w += v[q].w;
        }
        uint2 raw;
        raw.x = pack_bf16(__float2bfloat16_rn(a.x), __float2bfloat16_rn(a.y));
        raw.y = pack_bf16(__float2bfloat16_rn(a.z), __float2bfloat16_rn(a.w));
        const int tk = n0 + t;
        if (seg == 0) {
            *reinterpret_cast<float4*>(f.qhat + ((int64_t)tk * f.heads + head) * kHeadDim + 4 * lane) =
                norm_rope_q_regs(raw, w4, rh, f.eps, lane, f.rot);
        } else {
            const int64_t dst = ((int64_t)head * f.num_slots + cur.y) * kHeadDim + 4 * lane;
            if (seg == 1)
                *reinterpret_cast<uint2*>(f.K + dst) = norm_rope_k_regs(raw, w4, rh, rl, f.eps, lane, f.rot);
            else
                *reinterpret_cast<uint2*>(f.V + dst) = raw;  // v is written as given
        }
    };
    // two tokens a pass (t and t + 4): every load of both is in flight before the first is finished
    for (int t = t_lo + warp; t < t_hi; t += 8) {
        const int t2 = t + 4;
        const int2 c0 = tok[t - t_lo], c1 = t2 < t_hi ? tok[t2 - t_lo] : make_int2(-1, 0);
        float4 v0[NS], v1[NS];
        float2 h0[4], l0[4], h1[4], l1[4];
        if (c0.x >= 0) {
            partial(t, v0);
            rope_rows(c0.x, h0, l0);
        }
        if (c1.x >= 0) {
            partial(t2, v1);
            rope_rows(c1.x, h1, l1);
        }
        if (c0.x >= 0) finish(t, c0, v0, h0, l0);
        if (c1.x >= 0) finish(t2, c1, v1, h1, l1);
    }
}

// The segment holding output tile row m0: its tensor, its width and the tile's column in it.
__device__ __forceinline__ __nv_bfloat16* seg_of(const LinParams& p, int m0, int& width, int& col)
{
    const int s = m0 < p.seg_end[0] ? 0 : (m0 < p.seg_end[1] ? 1 : 2);
    const int start = s ? p.seg_end[s - 1] : 0;
    width = p.seg_end[s] - start;
    col = m0 - start;
    return p.y[s];
}

// Split-K epilogue of one CTA of a cluster of NS: sum its groups of four features
// [r * 32 / NS, (r + 1) * 32 / NS) of the tile over the NS partial tiles ([token][feature]
// fp32 in each CTA's shared memory at `local`), in rank order, and write them to y.  A
// thread issues the loads of up to 16 float4 (several items, every source) before the
// first sum, so the remote reads cost about one round trip rather than one per item.
template <int BN, int NS>
__device__ __forceinline__ void cluster_reduce(uint32_t local, int r, int tid, int n0, int tokens,
                                               __nv_bfloat16* y, int yw, int yc)
{
    constexpr int kPer = (kBM / 4) / NS;  // groups of four features per CTA
    constexpr int kPerThread = BN * kPer / kLinThreads;
    constexpr int R = (16 / NS) < kPerThread ? (16 / NS) : kPerThread;  // items per round
    static_assert(kPerThread % R == 0, "whole rounds");
    uint32_t src[NS];
#pragma unroll
    for (int q = 0; q < NS; ++q) src[q] = cluster_map(local, q);
#pragma unroll 1
    for (int r0 = 0; r0 < kPerThread; r0 += R) {
        float4 v[R][NS];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int idx = tid + kLinThreads * (r0 + u), t = idx / kPer, f = 4 * (r * kPer + idx % kPer);
            const uint32_t off = (uint32_t)(t * kBM + f) * 4;
#pragma unroll
            for (int q = 0; q < NS; ++q) v[u][q] = ld_cluster_f32x4(src[q] + off);
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int idx = tid + kLinThreads * (r0 + u), t = idx / kPer, f = 4 * (r * kPer + idx % kPer);
            float4 acc = v[u][0];
#pragma unroll
            for (int q = 1; q < NS; ++q) {
                acc.x += v[u][q].x;
                acc.y += v[u][q].y;
                acc.z += v[u][q].z;
                acc.w += v[u][q].w;
            }
            if (n0 + t < tokens) {
                uint2 o2;
                o2.x = pack_bf16(__float2bfloat16_rn(acc.x), __float2bfloat16_rn(acc.y));
                o2.y = pack_bf16(__float2bfloat16_rn(acc.z), __float2bfloat16_rn(acc.w));
                *reinterpret_cast<uint2*>(y + (int64_t)(n0 + t) * yw + yc + f) = o2;
            }
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(kLinThreads, BN == 64 ? 2 : 1)
    linear_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, LinParams p)
{
    using S = LinShape<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);
    const uint32_t bar_full = base + S::kBars, bar_empty = bar_full + 8 * S::kStages,
                   bar_done = bar_empty + 8 * S::kStages;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * BN, split = blockIdx.z;
    // this CTA's share of the input features, in whole 64-wide steps
    const int nk = p.in / kBK;
    const int k0 = (int)((int64_t)nk * split / p.splits), k1 = (int)((int64_t)nk * (split + 1) / p.splits);

    if (tid == 0) {
        for (int i = 0; i < 2 * S::kStages + 1; ++i) mbar_init(bar_full + 8 * i, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(base + S::kTmemSlot, BN);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + S::kTmemSlot);

    pdl_launch_dependents();  // the next projection may start streaming its weights
    if (warp == 0 && lane == 0) {
        // ---- producer: the W box (128 features x 64 inputs) and the x box (BN tokens x 64 inputs).
        // The first stages' weights are requested before waiting for the kernel before this one
        // (which may still be writing x); nothing this kernel writes is touched before the wait.
        const uint64_t pol_w = l2_policy_evict_first();  // each weight tile is read by one CTA per token tile
        const uint64_t pol_x = l2_policy_evict_last();   // x is read by every output tile
        const int early = min(k1 - k0, S::kStages);
        for (int i = 0; i < early; ++i) {
            const uint32_t a = base + i * S::kStageBytes, fb = bar_full + 8 * i;
            mbar_arrive_expect_tx(fb, S::kStageBytes);
            tma_load_2d(a, &tmW, (k0 + i) * kBK, m0, fb, pol_w);
        }
        pdl_wait();
        for (int i = 0; i < early; ++i)
            tma_load_2d(base + i * S::kStageBytes + S::kABytes, &tmX, (k0 + i) * kBK, n0, bar_full + 8 * i, pol_x);
        for (int k = k0 + early; k < k1; ++k) {
            const int i = k - k0, st = i % S::kStages;
            if (!mbar_wait(bar_empty + 8 * st, ((i / S::kStages) - 1) & 1)) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            const uint32_t a = base + st * S::kStageBytes, fb = bar_full + 8 * st;
            mbar_arrive_expect_tx(fb, S::kStageBytes);
            tma_load_2d(a, &tmW, k * kBK, m0, fb, pol_w);
            tma_load_2d(a + S::kABytes, &tmX, k * kBK, n0, fb, pol_x);
        }
    } else if (p.fused && warp >= 2) {
        // ---- the fused epilogue's token table (positions, validity, slots), while the product runs
        fused_tokens(p, reinterpret_cast<int2*>(sbase + S::kTok), BN, n0, m0, warp - 2, lane);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t idesc = umma_idesc_bf16(kBM, BN, 0, 0);
        for (int k = k0; k < k1; ++k) {
            const int i = k - k0, st = i % S::kStages;
            if (!mbar_wait_spin(bar_full + 8 * st, (i / S::kStages) & 1)) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t a = base + st * S::kStageBytes;
            const uint64_t da = umma_desc_sw128(a, 16, 1024), db = umma_desc_sw128(a + S::kABytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)  // 32 bytes further along K per step of 16
                umma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, i > 0 || kk > 0);
            umma_commit(bar_empty + 8 * st);
        }
        umma_commit(bar_done);  // also on a timeout: the epilogue and the release wait for it
    }
    __syncwarp();

    // ---- epilogue: thread (warp w, lane l) holds output feature m0 + 32 w + l for BN tokens
    pdl_wait();  // y may be read by the kernel before this one
    const bool ok = mbar_wait(bar_done, 0);
    tc_fence_after();
    int yw, yc;
    __nv_bfloat16* const y = seg_of(p, m0, yw, yc);
    const int o = yc + 32 * warp + lane;  // this thread's column of y
    if (p.splits == 1 && p.fused) {
        // stage the tile [token][feature] in the idle ring, then the token-major fused epilogue
        float* part = reinterpret_cast<float*>(sbase);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
            tmem_wait_ld_regs(v);
#pragma unroll
            for (int j = 0; j < 32; ++j) part[(c0 + j) * kBM + 32 * warp + lane] = ok ? __uint_as_float(v[j]) : 0.f;
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, BN);
        }
        if (ok) {
            const uint32_t none[1] = {0u};
            fused_rows<1>(p, none, part, reinterpret_cast<const int2*>(sbase + S::kTok), BN, n0, m0, warp, lane);
        }
        return;
    }
    if (p.splits == 1) {
        if (ok) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
                tmem_wait_ld_regs(v);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = n0 + c0 + j;
                    if (t < p.tokens) y[(int64_t)t * yw + o] = __float2bfloat16_rn(__uint_as_float(v[j]));
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, BN);
        }
        return;
    }
    // ---- split over the cluster: the partial tile, [token][feature] fp32, in this CTA's idle ring
    float* part = reinterpret_cast<float*>(sbase);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
        tmem_wait_ld_regs(v);
#pragma unroll
        for (int j = 0; j < 32; ++j) part[(c0 + j) * kBM + 32 * warp + lane] = ok ? __uint_as_float(v[j]) : 0.f;
    }
    tc_fence_before();
    cluster_sync();  // every partial tile of the cluster is in place
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, BN);
    }
    const uint32_t local = smem_u32(part);
    const int r = (int)cluster_rank();
    if (p.fused) {  // CTA r of the cluster finishes tokens [r BN / NS, (r + 1) BN / NS) of the tile
        auto run = [&](auto ns_tag) {
            constexpr int NS = decltype(ns_tag)::value;
            uint32_t src[NS];
#pragma unroll
            for (int q = 0; q < NS; ++q) src[q] = cluster_map(local, q);
            fused_rows<NS>(p, src, part, reinterpret_cast<const int2*>(sbase + S::kTok), BN, n0, m0, warp, lane);
        };
        switch (p.splits) {
        case 2: run(std::integral_constant<int, 2>{}); break;
        case 4: run(std::integral_constant<int, 4>{}); break;
        default: run(std::integral_constant<int, 8>{}); break;
        }
        cluster_sync();
        return;
    }
    switch (p.splits) {  // linear_splits gives 2, 4 or 8
    case 2: cluster_reduce<BN, 2>(local, r, tid, n0, p.tokens, y, yw, yc); break;
    case 4: cluster_reduce<BN, 4>(local, r, tid, n0, p.tokens, y, yw, yc); break;
    default: cluster_reduce<BN, 8>(local, r, tid, n0, p.tokens, y, yw, yc); break;
    }
    cluster_sync();  // no CTA leaves while another reads its shared memory
}

template <int BN>
cudaError_t launch_linear_bn(pkv_pool* pool, const void* x, const void* w, const LinParams& p, int splits,
                             cudaStream_t s)
{
    using S = LinShape<BN>;
    CUtensorMap tmW, tmX;
    if (!make_tmap_2d(&tmW, w, p.in, p.out, (uint64_t)p.in * 2, kBK, kBM) ||
        !make_tmap_2d(&tmX, x, p.in, p.tokens, (uint64_t)p.in * 2, kBK, BN))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(linear_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
    if (e != cudaSuccess) return e;
    const bool timed = pool->timer_on == 1;
    const int slot = timed ? (int)(pool->timer_count.fetch_add(1) % kTimerSlots) : 0;
    if (timed && (e = cudaEventRecord(pool->ev_start[slot], s)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.out / kBM, (p.tokens + BN - 1) / BN, splits);
    cfg.blockDim = dim3(kLinThreads);
    cfg.dynamicSmemBytes = S::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = splits;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = timed ? 0 : 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, linear_kernel<BN>, tmW, tmX, p);
    if (e != cudaSuccess) return e;
    if (timed && (e = cudaEventRecord(pool->ev_stop[slot], s)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

int linear_tile_tokens(int tokens) { return tokens <= 64 ? 64 : tokens <= 128 ? 128 : 256; }

// Split the input features over the CTAs of a cluster (at most 8) only while
// the output tiles leave resident CTA slots empty, keeping at least 4 steps of
// 64 input features per split.
int linear_splits(const pkv_pool* pool, int tokens, int in, int out)
{
    const int bn = linear_tile_tokens(tokens);
    const int tiles = (out / kBM) * ((tokens + bn - 1) / bn);
    const int slots = pool->num_sms * (bn == 64 ? 2 : 1);
    int splits = 1;
    while (splits < kMaxSplits && tiles * splits * 2 <= slots && (in / kBK) / (splits * 2) >= 4) splits *= 2;
    return splits;
}

static cudaError_t launch_linear_p(pkv_pool* pool, const void* x, const void* w, LinParams& p, cudaStream_t s)
{
    p.splits = linear_splits(pool, p.tokens, p.in, p.out);
    switch (linear_tile_tokens(p.tokens)) {
    case 64:
        return launch_linear_bn<64>(pool, x, w, p, p.splits, s);
    case 128:
        return launch_linear_bn<128>(pool, x, w, p, p.splits, s);
    default:
        return launch_linear_bn<256>(pool, x, w, p, p.splits, s);
    }
}

cudaError_t launch_linear(pkv_pool* pool, const void* x, const void* w, int tokens, int in, int nseg,
                          void* const* y, const int* widths, cudaStream_t s)
{
    LinParams p = {};
    int end = 0;
    for (int i = 0; i < 3; ++i) {
        end += i < nseg ? widths[i] : 0;
        p.y[i] = static_cast<__nv_bfloat16*>(i < nseg ? y[i] : nullptr);
        p.seg_end[i] = end;
    }
    p.err = pool->err;
    p.tokens = tokens;
    p.in = in;
    p.out = end;
    p.fused = 0;
    return launch_linear_p(pool, x, w, p, s);
}

cudaError_t launch_qkv_append(pkv_pool* pool, const void* x, const void* w_qkv, int tokens, int hidden,
                              const QkvAppend& a, cudaStream_t s)
{
    LinParams p = {};
    const int qw = pool->cfg.heads * kHeadDim, kw = pool->cfg.kv_heads * kHeadDim;
    p.seg_end[0] = qw;
    p.seg_end[1] = qw + kw;
    p.seg_end[2] = qw + 2 * kw;
    p.err = pool->err;
    p.tokens = tokens;
    p.in = hidden;
    p.out = p.seg_end[2];
    p.fused = 1;
    p.f.qw = static_cast<const __nv_bfloat16*>(a.q_norm_w);
    p.f.kw = static_cast<const __nv_bfloat16*>(a.k_norm_w);
    p.f.positions = a.positions;
    p.f.table = a.table;
    p.f.rope_hi = pool->rope_hi;
    p.f.rope_lo = pool->rope_lo;
    p.f.K = static_cast<__nv_bfloat16*>(pool->k);
    p.f.V = static_cast<__nv_bfloat16*>(pool->v);
    p.f.qhat = a.q_hat;
    p.f.num_slots = pool->num_slots;
    p.f.pages = a.pages;
    p.f.num_pages = pool->num_pages;
    p.f.max_seq = pool->cfg.max_seq;
    p.f.rot = pool->cfg.rotary_dim > 0 ? pool->cfg.rotary_dim : kHeadDim;
    p.f.heads = pool->cfg.heads;
    p.f.eps = static_cast<float>(pool->cfg.eps);
    return launch_linear_p(pool, x, w_qkv, p, s);
}

}  // namespace pkv
