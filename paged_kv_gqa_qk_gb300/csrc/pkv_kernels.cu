// Kernels of the paged-KV decode step (sm_103a).
//
//   prep_kernel        QK-norm + RoPE of q and k, page-slot append of k and v
//                      (one CTA per token).
//   attn_decode_kernel split-KV ("flash-decoding") attention over a token's
//                      pages: one CTA per (token, kv head, page range); TMA
//                      copies whole 16 KiB pages of K and V into a shared-
//                      memory ring, four consumer warps run QK^T and PV on
//                      mma.sync tensor cores with an online softmax.
//   combine_kernel     log-sum-exp merge of the page ranges of a token.
//
// Source of the computation: qwen3-8b Nest files, src/attention.linnet,
// GroupedQueryAttention.decode_paged / step_paged (q_norm/k_norm -> rope_rows
// -> page_slots + write_tokens -> paged_attention), src/norm.linnet (RmsNorm,
// eps 1e-6), src/rope.linnet (rotate-half tables, base 1e6).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr uint32_t kFull = 0xffffffffu;

// =====================================================================================
// G1: QK-norm + RoPE + KV append
// =====================================================================================
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
    const int32_t* table;           // [rows][pages]
    int P, rows, pages, num_pages, max_seq, heads, kv_heads;
    int64_t num_slots;
    float eps;
    const double2* rope;            // (cos, sin) [max_seq][64]
    __nv_bfloat16* K;               // [kv_heads][num_slots][128]
    __nv_bfloat16* V;
    float* qhat;                    // [tokens][heads][128]  normed + roped q
    int32_t* tok_len;               // [tokens]  attended length, 0 = skip
    int32_t* tok_row;               // [tokens]  table row
    uint32_t* err;
};

__device__ __forceinline__ void unpack4(uint2 r, float (&x)[4])
{
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xffff0000u);
}

// Round a double to bf16, nearest-even, with one rounding: truncate to fp32
// and mark inexactness in the last bit (round-to-odd; fp32 keeps 16 more bits
// than bf16), then round that to bf16.
__device__ __forceinline__ __nv_bfloat16 double_to_bf16_rn(double x)
{
    float f = __double2float_rz(x);
    if ((double)f != x) f = __uint_as_float(__float_as_uint(f) | 1u);
    return __float2bfloat16_rn(f);
}

__device__ __forceinline__ uint2 pack4(const float (&y)[4])
{
    uint2 r;
    r.x = pack_bf16(__float2bfloat16_rn(y[0]), __float2bfloat16_rn(y[1]));
    r.y = pack_bf16(__float2bfloat16_rn(y[2]), __float2bfloat16_rn(y[3]));
    return r;
}

// One CTA (4 warps) per token.  Lane l of a warp owns elements 4l..4l+3 of a
// head vector; the rotate-half partner of element i < 64 is element i + 64,
// held by lane l ^ 16.
__global__ void __launch_bounds__(128) prep_kernel(PrepParams p)
{
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

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
    // Every page the token will read must be a pool page.
    int bad = 0;
    const int32_t* trow = p.table + (int64_t)(row < 0 ? 0 : row) * p.pages;
    if (active && !e) {
        const int npg = pos / kPageSize + 1;
        for (int i = tid; i < npg; i += blockDim.x) {
            const int id = trow[i];
            bad |= (id < 0 || id >= p.num_pages);
        }
    }
    bad = __syncthreads_or(bad);
    if (active && !e && bad) e = PKV_DEVERR_PAGE;
    int64_t slot = 0;
    if (active && !e) {
        if (t < p.P && p.slots) {
            slot = p.slots[t];
            if (slot < 0 || slot >= p.num_slots) e = PKV_DEVERR_SLOT;
        } else {
            slot = (int64_t)trow[pos / kPageSize] * kPageSize + pos % kPageSize;
        }
    }
    if (!active || e) {
        if (tid == 0) {
            p.tok_len[t] = 0;
            p.tok_row[t] = 0;
            if (e) atomicOr(p.err, e);
        }
        return;
    }
    if (tid == 0) {
        p.tok_len[t] = pos + 1;
        p.tok_row[t] = row;
    }

    const int H = p.heads, G = p.kv_heads;
    const int fi = 4 * (lane & 15);  // frequency index of this lane's first element
    double cosd[4], sind[4];
    float cosv[4], sinv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const double2 cs = p.rope[(int64_t)pos * kRopeHalf + fi + i];
        cosd[i] = cs.x;
        sind[i] = cs.y;
        cosv[i] = (float)cs.x;
        sinv[i] = (float)cs.y;
    }
    float wq[4], wk[4];
    unpack4(*reinterpret_cast<const uint2*>(p.qw + 4 * lane), wq);
    unpack4(*reinterpret_cast<const uint2*>(p.kw + 4 * lane), wk);
    const float sgn = lane < 16 ? -1.f : 1.f;

    for (int task = warp; task < H + 2 * G; task += 4) {
        if (task < H + G) {
            const bool isq = task < H;
            const __nv_bfloat16* src = isq ? p.q + ((int64_t)t * H + task) * kHeadDim
                                           : p.k + ((int64_t)t * G + (task - H)) * kHeadDim;
            float x[4];
            unpack4(*reinterpret_cast<const uint2*>(src + 4 * lane), x);
            float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
            // RMSNorm over the head's 128 elements: x / sqrt(mean(x^2) + eps) * w,
            // then rotate-half RoPE: y*cos + rotate_half(y)*sin, rotate_half = (-y2, y1).
            // Both are linear in y, so the normaliser is applied last:
            //   r = inv * (u*cos -/+ u'*sin),  u = x*w  (exact in fp32: bf16 x bf16).
            const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
            float u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = x[i] * (isq ? wq[i] : wk[i]);
            if (isq) {
                float r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float partner = __shfl_xor_sync(kFull, u[i], 16);
                    r[i] = inv * (u[i] * cosv[i] + sgn * partner * sinv[i]);
                }
                *reinterpret_cast<float4*>(p.qhat + ((int64_t)t * H + task) * kHeadDim + 4 * lane) =
                    make_float4(r[0], r[1], r[2], r[3]);
            } else {
                // k is stored in bf16: rotate in double so cancellation between the
                // two terms cannot cost more than the final rounding
                __nv_bfloat16 r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float partner = __shfl_xor_sync(kFull, u[i], 16);
                    const double a = fma((double)(sgn * partner), sind[i], (double)u[i] * cosd[i]);
                    r[i] = double_to_bf16_rn(a * (double)inv);
                }
                const int g = task - H;
                *reinterpret_cast<uint2*>(p.K + ((int64_t)g * p.num_slots + slot) * kHeadDim + 4 * lane) =
                    make_uint2(pack_bf16(r[0], r[1]), pack_bf16(r[2], r[3]));
            }
        } else {
            const int g = task - H - G;  // v is written as given
            const uint2 raw = *reinterpret_cast<const uint2*>(p.v + ((int64_t)t * G + g) * kHeadDim + 4 * lane);
            *reinterpret_cast<uint2*>(p.V + ((int64_t)g * p.num_slots + slot) * kHeadDim + 4 * lane) = raw;
        }
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
    p.num_slots = pool->num_slots;
    p.eps = static_cast<float>(pool->cfg.eps);
    p.rope = pool->rope;
    p.K = static_cast<__nv_bfloat16*>(pool->k);
    p.V = static_cast<__nv_bfloat16*>(pool->v);
    p.qhat = reinterpret_cast<float*>(a.ws + plan.off_qhat);
    p.tok_len = reinterpret_cast<int32_t*>(a.ws + plan.off_len);
    p.tok_row = reinterpret_cast<int32_t*>(a.ws + plan.off_row);
    p.err = pool->err;
    prep_kernel<<<plan.tokens, 128, 0, s>>>(p);
    return cudaGetLastError();
}

// =====================================================================================
// G2: split-KV decode attention
// =====================================================================================
//
// CTA (token t, kv head g, split s) attends the 4 query heads of kv head g
// over pages [s*chunk, min(npages, (s+1)*chunk)) of the token's row.
//
// Warp roles: warps 0-3 consume, warp 4 produces.  The producer streams the
// pages through a ring of kStages stages; each stage is one page of K and one
// of V for kv head g, each copied as two 64x64 boxes (head-dim halves) with
// 128-byte swizzle, so ldmatrix reads them without bank conflicts.
//
// Consumer warp w takes positions 16w..16w+15 of every page.
//   QK^T:  S[16 pos][8 cols] = K_tile[16 pos][128] * Qb[128][8 cols]
//          cols 0-3 = bf16 head of q (heads 4g..4g+3, scaled by log2(e)/sqrt(128)),
//          cols 4-7 = bf16 of the remainder: S = col h + col h+4 carries q to
//          ~16 bits, so the logits keep fp32-level accuracy.
//   PV:    O^T[128 dims][8 cols] += V_tile^T[128][16 pos] * Pb[16 pos][8 cols]
//          cols 0-3 = bf16(p), cols 4-7 = bf16(p - bf16(p)); O = col h + col h+4.
// The softmax is kept per warp (running max m and sum l per head, base 2);
// the four warps' (m, l, O) are merged through shared memory at the end.
struct AttnParams {
    const float* qhat;       // [tokens][heads][128]
    const int32_t* tok_len;  // [tokens]
    const int32_t* tok_row;  // [tokens]
    const int32_t* table;    // [rows][pages]
    int pages, chunk, max_splits, heads, kv_heads;
    __nv_bfloat16* out;      // [tokens][heads][128]
    float* part_o;           // [tokens][heads][max_splits][128]
    float* part_lse;         // [tokens][heads][max_splits]   (base-2 log-sum-exp)
    uint32_t* err;
};

constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = 4 * 8192;  // K lo, K hi, V lo, V hi

template <int kStages>
struct AttnSmem {
    static constexpr int kRing = kStages * kStageBytes;
    static constexpr int kMergeO = kRing;                                   // float [4 warps][4 heads][128]
    static constexpr int kMergeM = kMergeO + kConsumerWarps * 4 * 128 * 4;  // float [4][4]
    static constexpr int kMergeL = kMergeM + 64;                            // float [4][4]
    static constexpr int kBars = kMergeL + 64;                              // uint64 full[kStages], empty[kStages]
    static constexpr int kFlag = kBars + 2 * 8 * kStages;
    static constexpr int kBytes = kFlag + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
};

template <int kStages>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       AttnParams p)
{
    using L = AttnSmem<kStages>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);
    const uint32_t bar_full = base + L::kBars;
    const uint32_t bar_empty = bar_full + 8 * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + L::kFlag);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lin = blockIdx.x;
    const int s = lin % p.max_splits;
    const int tg = lin / p.max_splits;
    const int g = tg % p.kv_heads;
    const int t = tg / p.kv_heads;
    const int H = p.heads;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();
    pdl_wait();  // everything below reads what the prep kernel wrote

    const int len = p.tok_len[t];
    if (len == 0) {  // skipped token: split 0 writes zeros for this kv head's query heads
        if (s == 0) {
            for (int i = tid; i < kGroup * kHeadDim / 4; i += kAttnThreads) {
                const int h = i / (kHeadDim / 4), d = 4 * (i % (kHeadDim / 4));
                *reinterpret_cast<uint2*>(p.out + ((int64_t)t * H + g * kGroup + h) * kHeadDim + d) =
                    make_uint2(0u, 0u);
            }
        }
        return;
    }
    const int npg = (len + kPageSize - 1) / kPageSize;
    const int nsplit = (npg + p.chunk - 1) / p.chunk;
    if (s >= nsplit) return;
    const int pg0 = s * p.chunk;
    const int n = min(npg, pg0 + p.chunk) - pg0;
    const int row = p.tok_row[t];

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------------ producer
        const int32_t* trow = p.table + (int64_t)row * p.pages + pg0;
        const uint64_t pol = l2_policy_evict_first();
        int issued = 0;
        bool ok = true;
        for (int b0 = 0; b0 < n && ok; b0 += 32) {
            const int mine = (b0 + lane < n) ? trow[b0 + lane] : 0;
            const int cnt = min(32, n - b0);
            for (int j = 0; j < cnt; ++j) {
                const int i = b0 + j;
                const int page = __shfl_sync(kFull, mine, j);
                const int st = i % kStages;
                if (i >= kStages) {
                    if (!mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1) || *abort_flag) {
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) {
                    const uint32_t dst = base + st * kStageBytes;
                    const uint32_t fb = bar_full + 8 * st;
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    const int y = page * kPageSize;
                    tma_load_3d(dst, &tmK, 0, y, g, fb, pol);
                    tma_load_3d(dst + 8192, &tmK, 64, y, g, fb, pol);
                    tma_load_3d(dst + 16384, &tmV, 0, y, g, fb, pol);
                    tma_load_3d(dst + 24576, &tmV, 64, y, g, fb, pol);
                }
                ++issued;
                __syncwarp();
            }
        }
        if (!ok) {
            if (lane == 0) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
                // wait (bounded) for the copies still in flight before the CTA exits
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(bar_full + 8 * (i % kStages), (i / kStages) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------------------------- consumers
    const int gid = lane >> 2, tig = lane & 3;
    // B fragments of q: col n = gid -> head gid&3, part gid>>2 (0 head, 1 remainder)
    uint32_t bq[8][2];
    {
        const int hh = gid & 3;
        const bool rem = gid >= 4;
        const float* qh = p.qhat + ((int64_t)t * H + g * kGroup + hh) * kHeadDim;
        const float sc = 1.4426950408889634f * 0.088388347648318440f;  // log2(e) / sqrt(128)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int d0 = 16 * ks + 2 * tig;
            const float2 xa = *reinterpret_cast<const float2*>(qh + d0);
            const float2 xb = *reinterpret_cast<const float2*>(qh + d0 + 8);
            const float xs[4] = {xa.x * sc, xa.y * sc, xb.x * sc, xb.y * sc};
            __nv_bfloat16 hd[4], tl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) split_bf16(xs[i], hd[i], tl[i]);
            bq[ks][0] = rem ? pack_bf16(tl[0], tl[1]) : pack_bf16(hd[0], hd[1]);
            bq[ks][1] = rem ? pack_bf16(tl[2], tl[3]) : pack_bf16(hd[2], hd[3]);
        }
    }

    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float mA = -CUDART_INF_F, mB = -CUDART_INF_F, lA = 0.f, lB = 0.f;
    const bool rem_lane = tig >= 2;  // this lane's S/O columns are the remainder columns
    // source lanes of the P fragment (see the PV comment above)
    const int hh = gid & 3, prt = gid >> 2;
    const int srcA = 4 * (2 * tig) + (hh >> 1) + 2 * prt;
    const int srcB = srcA + 4;
    const int r_ld = lane & 7, j_ld = lane >> 3;
    bool ok = true;

    for (int i = 0; i < n; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(bar_full + 8 * st, (i / kStages) & 1)) {
            ok = false;
            break;
        }
        const uint32_t kb = base + st * kStageBytes;
        const uint32_t vb = kb + 16384;

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
        const int pbase = (pg0 + i) * kPageSize + 16 * warp;
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
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
    if (!ok) {
        if (lane == 0) {
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    // ---- per-warp finish: full sums over the warp's positions, head + remainder columns
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
        lA += __shfl_xor_sync(kFull, lA, o2);
        lB += __shfl_xor_sync(kFull, lB, o2);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[mt][k] += __shfl_xor_sync(kFull, o[mt][k], 2);

    float* sO = reinterpret_cast<float*>(sbase + L::kMergeO);
    float* sM = reinterpret_cast<float*>(sbase + L::kMergeM);
    float* sL = reinterpret_cast<float*>(sbase + L::kMergeL);
    if (tig < 2) {
        const int hA = 2 * tig, hB = hA + 1;
        float* oA = sO + (warp * 4 + hA) * kHeadDim;
        float* oB = sO + (warp * 4 + hB) * kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = 16 * mt + gid;
            oA[d] = o[mt][0];
            oB[d] = o[mt][1];
            oA[d + 8] = o[mt][2];
            oB[d + 8] = o[mt][3];
        }
        if (gid == 0) {
            sM[warp * 4 + hA] = mA;
            sM[warp * 4 + hB] = mB;
            sL[warp * 4 + hA] = lA;
            sL[warp * 4 + hB] = lB;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if (*abort_flag) return;

    // ---- merge the four warps: thread -> (head h, dims 4c..4c+3)
    {
        const int h = tid >> 5, c = tid & 31;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sM[w * 4 + h]);
        float Ls = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = sM[w * 4 + h];
            const float f = (mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
            Ls += f * sL[w * 4 + h];
            const float4 ow = *reinterpret_cast<const float4*>(sO + (w * 4 + h) * kHeadDim + 4 * c);
            acc[0] += f * ow.x;
            acc[1] += f * ow.y;
            acc[2] += f * ow.z;
            acc[3] += f * ow.w;
        }
        const float inv = 1.f / Ls;
        const int qh = g * kGroup + h;
        if (nsplit == 1) {
            const float y[4] = {acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv};
            *reinterpret_cast<uint2*>(p.out + ((int64_t)t * H + qh) * kHeadDim + 4 * c) = pack4(y);
        } else {
            const int64_t ph = ((int64_t)t * H + qh) * p.max_splits + s;
            *reinterpret_cast<float4*>(p.part_o + ph * kHeadDim + 4 * c) =
                make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            if (c == 0) p.part_lse[ph] = M + log2f(Ls);
        }
    }
}

constexpr int kDecodeStages = 3;

cudaError_t configure_kernels()
{
    return cudaFuncSetAttribute(attn_decode_kernel<kDecodeStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnSmem<kDecodeStages>::kAlloc);
}

cudaError_t launch_attn_decode(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s)
{
    using L = AttnSmem<kDecodeStages>;
    AttnParams p;
    p.qhat = reinterpret_cast<const float*>(a.ws + plan.off_qhat);
    p.tok_len = reinterpret_cast<const int32_t*>(a.ws + plan.off_len);
    p.tok_row = reinterpret_cast<const int32_t*>(a.ws + plan.off_row);
    p.table = a.table;
    p.pages = a.pages;
    p.chunk = plan.chunk;
    p.max_splits = plan.max_splits;
    p.heads = pool->cfg.heads;
    p.kv_heads = pool->cfg.kv_heads;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.part_o = reinterpret_cast<float*>(a.ws + plan.off_po);
    p.part_lse = reinterpret_cast<float*>(a.ws + plan.off_plse);
    p.err = pool->err;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)plan.tokens * pool->cfg.kv_heads * plan.max_splits));
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_decode_kernel<kDecodeStages>, pool->tmap_k, pool->tmap_v, p);
}

// =====================================================================================
// G3: log-sum-exp combine of the splits
// =====================================================================================
struct CombineParams {
    const int32_t* tok_len;
    int chunk, max_splits, heads;
    const float* part_o;
    const float* part_lse;
    __nv_bfloat16* out;
};

// One warp per (token, query head); lane owns dims 4*lane..4*lane+3.
//   out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M)
__global__ void __launch_bounds__(128) combine_kernel(CombineParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = p.heads / 4;
    const int t = blockIdx.x / hq;
    const int h = (blockIdx.x % hq) * 4 + warp;
    pdl_wait();
    const int len = p.tok_len[t];
    if (len == 0) return;
    const int npg = (len + kPageSize - 1) / kPageSize;
    const int nsplit = (npg + p.chunk - 1) / p.chunk;
    if (nsplit <= 1) return;
    const int64_t ph = ((int64_t)t * p.heads + h) * p.max_splits;
    const float* lse = p.part_lse + ph;
    float M = -CUDART_INF_F;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o2));
    float wsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < nsplit; ++s) {
        const float w = exp2f(lse[s] - M);
        const float4 o = *reinterpret_cast<const float4*>(p.part_o + (ph + s) * kHeadDim + 4 * lane);
        wsum += w;
        acc[0] += w * o.x;
        acc[1] += w * o.y;
        acc[2] += w * o.z;
        acc[3] += w * o.w;
    }
    const float inv = 1.f / wsum;
    const float y[4] = {acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv};
    *reinterpret_cast<uint2*>(p.out + ((int64_t)t * p.heads + h) * kHeadDim + 4 * lane) = pack4(y);
}

cudaError_t launch_combine(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s)
{
    if (plan.max_splits <= 1) return cudaSuccess;
    CombineParams p;
    p.tok_len = reinterpret_cast<const int32_t*>(a.ws + plan.off_len);
    p.chunk = plan.chunk;
    p.max_splits = plan.max_splits;
    p.heads = pool->cfg.heads;
    p.part_o = reinterpret_cast<const float*>(a.ws + plan.off_po);
    p.part_lse = reinterpret_cast<const float*>(a.ws + plan.off_plse);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(plan.tokens * (pool->cfg.heads / 4)));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace pkv
