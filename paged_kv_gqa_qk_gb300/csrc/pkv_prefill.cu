// Prompt-chunk attention of step_paged on tcgen05 tensor cores (sm_103a).
//
// qwen3-8b Nest files, src/attention.linnet, GroupedQueryAttention.step_paged
// (and prefill_paged): after every token of the call has been written to the
// pool (prep_kernel), prompt token p attends over table[rows[p]] for
// positions 0..positions[p] -- its own chunk's earlier keys included.
//
// A CTA takes a tile of 32 consecutive prompt tokens and one kv head g.  The
// 4 query heads of g times the 32 tokens are the M = 128 rows of the matrix
// products, row m = head (m / 32) of the group, token (m % 32) of the tile, so
// tensor-memory lane m belongs to thread m of the four softmax warps.  For
// every page j of the row (up to the tile's last position):
//   S_j  = Q K_j^T           128 x 64,  K = 128 dims   (tcgen05, into TMEM)
//   P_j  = 2^(S_j - m)       causal mask, online max m (softmax warps, bf16 to smem)
//   O   += P_j V_j           128 x 128, K = 64 positions (tcgen05, into TMEM)
// Q carries the QK-norm, the RoPE and the score scale log2(e)/sqrt(128), so S
// is in base-2 units.  The running max is only moved (and O, l rescaled in
// place) when a page raises it by more than 8: in between, P stays below 2^8.
//
// Warp roles: 0-3 softmax (and the q preparation and the epilogue), 4 TMA
// producer (pages of K and V through a 3-stage ring, the layout the decode
// kernel also uses), 5 tensor-memory allocation and the MMA-issuing thread.
// S is double-buffered in tensor memory and P in shared memory, so the
// products of page j+1 overlap the softmax of page j.
//
// A tile whose tokens belong to several table rows (where one prompt ends and
// the next begins) is processed once per row; tokens of the other rows are
// masked out of that pass.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {

constexpr uint32_t kAll = 0xffffffffu;
constexpr int kTileTok = 32;                 // prompt tokens per tile
constexpr int kTileRows = kTileTok * kGroup;  // 128 = M
constexpr int kPfStages = 3;
constexpr int kPfStageBytes = 4 * 8192;      // K lo, K hi, V lo, V hi (one page, one kv head)
constexpr int kPfThreads = 6 * 32;
constexpr int kSoftmaxWarps = 4, kProducer = 4, kIssuer = 5;
constexpr uint32_t kTmemCols = 256;          // S buffers at columns 0 and 64, O at 128..255
constexpr float kRescale = 8.f;              // log2 headroom before the running max moves

struct PfSmem {
    static constexpr int kQ = 0;                                  // bf16 [2 halves][128 rows][128 B], swizzled
    static constexpr int kRing = kQ + 2 * kTileRows * 128;        // stages x 32 KiB
    static constexpr int kP = kRing + kPfStages * kPfStageBytes;  // bf16 [2 buffers][128 rows][128 B]
    static constexpr int kTok = kP + 2 * kTileRows * 128;         // int pos[32], row[32]
    static constexpr int kRuns = kTok + 2 * kTileTok * 4;         // int row[32], npages[32], count
    static constexpr int kW = kRuns + (2 * kTileTok + 4) * 4;     // bf16 q_norm weights [128]
    static constexpr int kBars = kW + 256;
    // full[S], empty[S], s_ready[2], p_ready[2], o_done[2], epi_done
    static constexpr int kNumBars = 2 * kPfStages + 7;
    static constexpr int kTmemSlot = kBars + 8 * kNumBars;
    static constexpr int kFlag = kTmemSlot + 16;
    static constexpr int kBytes = kFlag + 16;
    static constexpr int kAlloc = kBytes + 1024;
};

// byte offset of element c (< 64) of row r in a [rows][64 bf16] tile with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2; }

struct PfParams {
    const __nv_bfloat16* q;   // [P + rows][heads][128], prompt tokens first
    const __nv_bfloat16* qw;  // q_norm weights [128]
    const int32_t* tok_len;   // [P] attended length from prep_kernel, 0 = skip
    const int32_t* tok_row;   // [P]
    const int32_t* table;     // [rows][pages]
    const float2* rope_hi;    // (cos, sin) [max_seq][64]
    __nv_bfloat16* out;       // [P + rows][heads][128]
    uint32_t* err;
    int P, pages, heads, kv_heads, ntiles;
    float eps;
};

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, PfParams p)
{
    using L = PfSmem;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw_base);
    const uint32_t bar0 = base + L::kBars;
    const uint32_t bar_full = bar0, bar_empty = bar0 + 8 * kPfStages;
    const uint32_t bar_s = bar0 + 16 * kPfStages, bar_p = bar_s + 16, bar_o = bar_p + 16, bar_epi = bar_o + 16;
    int* sPos = reinterpret_cast<int*>(sbase + L::kTok);
    int* sRow = sPos + kTileTok;
    int* sRunRow = reinterpret_cast<int*>(sbase + L::kRuns);
    int* sRunPages = sRunRow + kTileTok;
    int* sNumRuns = sRunPages + kTileTok;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + L::kFlag);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x % p.ntiles, g = blockIdx.x / p.ntiles;
    const int p0 = tile * kTileTok;

    if (tid == 0) {
        for (int i = 0; i < 2 * kPfStages; ++i) mbar_init(bar0 + 8 * i, 1);  // full (producer), empty (commit)
        mbar_init(bar_s, 1);
        mbar_init(bar_s + 8, 1);
        mbar_init(bar_p, kSoftmaxWarps);
        mbar_init(bar_p + 8, kSoftmaxWarps);
        mbar_init(bar_o, 1);
        mbar_init(bar_o + 8, 1);
        mbar_init(bar_epi, kSoftmaxWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kIssuer) tmem_alloc(base + L::kTmemSlot, kTmemCols);
    if (warp == kProducer && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    pdl_wait();  // prep_kernel's appends and token table

    // ---- the tile's tokens, and its runs (one per table row among its valid tokens)
    if (tid < kTileTok) {
        const int t = p0 + tid;
        const int len = t < p.P ? p.tok_len[t] : 0;
        sPos[tid] = len - 1;  // -1: not a token, or skipped
        sRow[tid] = len > 0 ? p.tok_row[t] : -1;
    } else if (tid < 2 * kTileTok) {
        reinterpret_cast<uint2*>(sbase + L::kW)[tid - kTileTok] = reinterpret_cast<const uint2*>(p.qw)[tid - kTileTok];
    }
    __syncthreads();
    if (tid == 0) {
        int nr = 0;
        for (int i = 0; i < kTileTok; ++i) {
            if (sPos[i] < 0) continue;
            int r = 0;
            while (r < nr && sRunRow[r] != sRow[i]) ++r;
            if (r == nr) {
                sRunRow[nr] = sRow[i];
                sRunPages[nr] = 0;
                ++nr;
            }
            sRunPages[r] = max(sRunPages[r], sPos[i] / kPageSize + 1);
        }
        *sNumRuns = nr;
    }

    // ---- Q: QK-norm + RoPE of (head 4g + warp, token lane), scaled by log2(e)/sqrt(128), bf16
    if (warp < kSoftmaxWarps) {
        const int m = tid;  // tile row
        const int pos = sPos[lane];
        uint8_t* q0 = sbase + L::kQ;
        if (pos >= 0) {
            // two passes over the row (the second from L1): sum of squares, then norm + rotate
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q + ((int64_t)(p0 + lane) * p.heads + g * kGroup + warp) * kHeadDim);
            const uint4* wsm = reinterpret_cast<const uint4*>(sbase + L::kW);
            const float2* rp = p.rope_hi + (int64_t)pos * kRopeHalf;
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < kHeadDim / 8; ++c) {
                const uint4 r = src[c];
                const uint32_t rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = __uint_as_float(rv[e] << 16), b = __uint_as_float(rv[e] & 0xffff0000u);
                    ss += a * a + b * b;
                }
            }
            const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps) * (1.4426950408889634f * 0.088388347648318440f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // dims 8c..8c+7 of the first half and their partners 64 apart
                const uint4 rl = src[c], rh = src[c + 8], wl = wsm[c], wh = wsm[c + 8];
                const uint32_t xl[4] = {rl.x, rl.y, rl.z, rl.w}, xh[4] = {rh.x, rh.y, rh.z, rh.w};
                const uint32_t vl[4] = {wl.x, wl.y, wl.z, wl.w}, vh[4] = {wh.x, wh.y, wh.z, wh.w};
                uint32_t lo[4], hi[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float y[2], z[2];
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int d = 8 * c + 2 * e + b;
                        const float ul = __uint_as_float(b ? (xl[e] & 0xffff0000u) : (xl[e] << 16)) *
                                         __uint_as_float(b ? (vl[e] & 0xffff0000u) : (vl[e] << 16));
                        const float uh = __uint_as_float(b ? (xh[e] & 0xffff0000u) : (xh[e] << 16)) *
                                         __uint_as_float(b ? (vh[e] & 0xffff0000u) : (vh[e] << 16));
                        const float2 cs = rp[d];
                        y[b] = inv * (ul * cs.x - uh * cs.y);  // y[d]      = u[d] cos - u[d+64] sin
                        z[b] = inv * (uh * cs.x + ul * cs.y);  // y[d + 64] = u[d+64] cos + u[d] sin
                    }
                    lo[e] = pack_bf16(__float2bfloat16_rn(y[0]), __float2bfloat16_rn(y[1]));
                    hi[e] = pack_bf16(__float2bfloat16_rn(z[0]), __float2bfloat16_rn(z[1]));
                }
                *reinterpret_cast<uint4*>(q0 + sw128(m, 8 * c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4*>(q0 + kTileRows * 128 + sw128(m, 8 * c)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4*>(q0 + sw128(m, 8 * c)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(q0 + kTileRows * 128 + sw128(m, 8 * c)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q is read by the tensor cores
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + L::kTmemSlot);
    const int nruns = *sNumRuns;

    if (warp == kProducer) {
        // ================================================================ producer
        const uint64_t pol = l2_policy_evict_last();  // a prompt's tiles re-read the same pages
        int i = 0;
        bool ok = true;
        for (int r = 0; r < nruns && ok; ++r) {
            const int row = sRunRow[r];
            const int n = sRunPages[r];
            for (int b0 = 0; b0 < n && ok; b0 += 32) {
                const int mine = (b0 + lane < n) ? page_of(p.table, p.pages, row, b0 + lane) : 0;
                for (int jj = 0; jj < min(32, n - b0); ++jj, ++i) {
                    const int page = __shfl_sync(kAll, mine, jj);
                    const int st = i % kPfStages;
                    if (i >= kPfStages && (!mbar_wait(bar_empty + 8 * st, ((i / kPfStages) - 1) & 1) || *abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t fb = bar_full + 8 * st, dst = base + L::kRing + st * kPfStageBytes;
                        mbar_arrive_expect_tx(fb, kPfStageBytes);
                        const int y = page * kPageSize;
                        tma_load_3d(dst, &tmK, 0, y, g, fb, pol);
                        tma_load_3d(dst + 8192, &tmK, 64, y, g, fb, pol);
                        tma_load_3d(dst + 16384, &tmV, 0, y, g, fb, pol);
                        tma_load_3d(dst + 24576, &tmV, 64, y, g, fb, pol);
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
            for (int k = max(0, i - kPfStages); k < i; ++k)
                mbar_wait(bar_full + 8 * (k % kPfStages), (k / kPfStages) & 1);
        }
    } else if (warp == kIssuer) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = umma_idesc_bf16(kTileRows, kPageSize, 0, 0);
            constexpr uint32_t id_pv = umma_idesc_bf16(kTileRows, kHeadDim, 0, 1);
            const uint32_t qb = base + L::kQ, pb = base + L::kP;
            bool ok = true;
            int jg = 0;
            for (int r = 0; r < nruns && ok; ++r) {
                const int n = sRunPages[r];
                for (int jj = 0; jj <= n && ok; ++jj) {
                    if (jj < n) {  // S_j = Q K_j^T
                        const int j = jg + jj, st = j % kPfStages, sb = j & 1;
                        if (!mbar_wait(bar_full + 8 * st, (j / kPfStages) & 1) || *abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t kst = base + L::kRing + st * kPfStageBytes;
#pragma unroll
                        for (int k = 0; k < kHeadDim / 16; ++k) {
                            const uint64_t a = umma_desc_sw128(qb + (k >> 2) * (kTileRows * 128) + (k & 3) * 32, 16, 1024);
                            const uint64_t b = umma_desc_sw128(kst + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
                            umma_bf16(tmem + sb * kPageSize, a, b, id_qk, k > 0);
                        }
                        umma_commit(bar_s + 8 * sb);
                    }
                    if (jj >= 1) {  // O += P_{j-1} V_{j-1}
                        const int j = jg + jj - 1, st = j % kPfStages, sb = j & 1;
                        if (!mbar_wait(bar_p + 8 * sb, (j >> 1) & 1) ||
                            (jj == 1 && r > 0 && !mbar_wait(bar_epi, (r - 1) & 1)) || *abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t vst = base + L::kRing + st * kPfStageBytes + 16384;
#pragma unroll
                        for (int k = 0; k < kPageSize / 16; ++k) {
                            const uint64_t a = umma_desc_sw128(pb + sb * (kTileRows * 128) + k * 32, 16, 1024);
                            const uint64_t b = umma_desc_sw128(vst + k * 2048, 8192, 1024);
                            umma_bf16(tmem + 2 * kPageSize, a, b, id_pv, jj > 1 || k > 0);
                        }
                        umma_commit(bar_o + 8 * sb);
                        umma_commit(bar_empty + 8 * st);
                    }
                }
                jg += n;
            }
            if (!ok) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax warps
        const int m = tid;                 // tile row: head `warp` of the group, token `lane`
        const int pos = sPos[lane];
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        uint8_t* pbuf = sbase + L::kP;
        bool ok = true;
        int jg = 0;
        for (int r = 0; r < nruns && ok; ++r) {
            const int n = sRunPages[r];
            const bool active = pos >= 0 && sRow[lane] == sRunRow[r];
            float m_used = -CUDART_INF_F, l = 0.f;
            for (int jj = 0; jj < n; ++jj) {
                const int j = jg + jj, sb = j & 1;
                if (!mbar_wait(bar_s + 8 * sb, (j >> 1) & 1) || *abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[kPageSize];
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tl + sb * kPageSize, v0);
                    tmem_ld32(tl + sb * kPageSize + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        s[c] = __uint_as_float(v0[c]);
                        s[c + 32] = __uint_as_float(v1[c]);
                    }
                }
                // causal mask: keys up to pos; only a page that reaches past pos needs it
                const int first = jj * kPageSize;
                if (!active || first > pos) {
#pragma unroll
                    for (int c = 0; c < kPageSize; ++c) s[c] = -CUDART_INF_F;
                } else if (first + kPageSize - 1 > pos) {
#pragma unroll
                    for (int c = 0; c < kPageSize; ++c)
                        if (first + c > pos) s[c] = -CUDART_INF_F;
                }
                float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int c = 4; c < kPageSize; c += 4) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx4[e] = fmaxf(mx4[e], s[c + e]);
                }
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                // move the running max (rescaling O and l) only when this page raises it by > 8
                bool need = false;
                float alpha = 1.f;
                if (jj == 0) {
                    m_used = mx;
                } else if (mx > m_used + kRescale) {
                    need = true;
                    alpha = exp2f(m_used - mx);
                }
                if (__any_sync(kAll, need)) {
                    const int jp = j - 1;  // O must hold the previous page's product first
                    if (!mbar_wait(bar_o + 8 * (jp & 1), (jp >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kHeadDim; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tl + 2 * kPageSize + c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st16(tl + 2 * kPageSize + c, v);
                    }
                    tmem_wait_st();
                    if (need) {
                        l *= alpha;
                        m_used = mx;
                    }
                }
                // P_j = 2^(S_j - m): into P buffer sb once the product two pages back has read it
                // (a row with no key yet has m = -inf: its p are all 0)
                const float msub = m_used == -CUDART_INF_F ? 0.f : m_used;
                float ps4[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[kPageSize / 2];
#pragma unroll
                for (int c = 0; c < kPageSize; c += 2) {
                    const float a = ex2_approx(s[c] - msub);
                    const float b = ex2_approx(s[c + 1] - msub);
                    ps4[(c >> 1) & 3] += a + b;
                    __nv_bfloat162 ab = __floats2bfloat162_rn(a, b);
                    pk[c / 2] = *reinterpret_cast<uint32_t*>(&ab);
                }
                l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
                if (j >= 2 && !mbar_wait(bar_o + 8 * sb, ((j - 2) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t* prow = pbuf + sb * (kTileRows * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(prow + sw128(m, 8 * c)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P is read by the tensor cores
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p + 8 * sb);
            }
            if (!ok) break;
            // ---- epilogue of this row's pass: O / l for the active rows
            const int jl = jg + n - 1;
            if (!mbar_wait(bar_o + 8 * (jl & 1), (jl >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            __nv_bfloat16* dst = p.out + ((int64_t)(p0 + lane) * p.heads + g * kGroup + warp) * kHeadDim;
            const float inv = active ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < kHeadDim; c += 16) {
                uint32_t v[16];
                tmem_ld16(tl + 2 * kPageSize + c, v);
                tmem_wait_ld();
                if (active) {
                    uint32_t o8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        o8[e] = pack_bf16(__float2bfloat16_rn(__uint_as_float(v[2 * e]) * inv),
                                          __float2bfloat16_rn(__uint_as_float(v[2 * e + 1]) * inv));
                    *reinterpret_cast<uint4*>(dst + c) = make_uint4(o8[0], o8[1], o8[2], o8[3]);
                    *reinterpret_cast<uint4*>(dst + c + 8) = make_uint4(o8[4], o8[5], o8[6], o8[7]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_epi);
            jg += n;
        }
        // skipped tokens of the tile: zero output
        if (pos < 0 && p0 + lane < p.P) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(p0 + lane) * p.heads + g * kGroup + warp) * kHeadDim);
#pragma unroll
            for (int c = 0; c < kHeadDim / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kIssuer) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t configure_prefill()
{
    return cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem::kAlloc);
}

cudaError_t launch_prefill(const pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s)
{
    PfParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.qw = static_cast<const __nv_bfloat16*>(a.q_norm_w);
    p.tok_len = reinterpret_cast<const int32_t*>(a.ws + plan.off_len);
    p.tok_row = reinterpret_cast<const int32_t*>(a.ws + plan.off_row);
    p.table = a.table;
    p.rope_hi = pool->rope_hi;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.err = pool->err;
    p.P = a.P;
    p.pages = a.pages;
    p.heads = pool->cfg.heads;
    p.kv_heads = pool->cfg.kv_heads;
    p.ntiles = (a.P + kTileTok - 1) / kTileTok;
    p.eps = static_cast<float>(pool->cfg.eps);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.ntiles * p.kv_heads));
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = PfSmem::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel, pool->tmap_k, pool->tmap_v, p);
}

}  // namespace pkv
