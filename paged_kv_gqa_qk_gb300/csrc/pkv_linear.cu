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
// input features are split over `splits` CTAs that write fp32 partial tiles
// to the workspace, and a second kernel sums them in a fixed order.
#include <cuda_bf16.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {

constexpr int kLinThreads = 128;
constexpr int kBM = 128;         // output features per tile (M)
constexpr int kBK = 64;          // input features per ring stage (one 128-byte swizzle span)
constexpr int kLinSmem = 192 * 1024;

template <int BN>
struct LinShape {
    static constexpr int kABytes = kBM * kBK * 2;  // 16 KiB of W
    static constexpr int kBBytes = BN * kBK * 2;   // x
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = kLinSmem / kStageBytes;
    static constexpr int kBars = kStages * kStageBytes;  // full[S], empty[S], done
    static constexpr int kTmemSlot = kBars + 8 * (2 * kStages + 1);
    static constexpr int kAlloc = kTmemSlot + 16 + 1024;
};

struct LinParams {
    __nv_bfloat16* y;   // [tokens][out], when splits == 1
    float* part;        // [splits][tokens][out], when splits > 1
    uint32_t* err;
    int tokens, in, out, splits;
};

template <int BN>
__global__ void __launch_bounds__(kLinThreads, 1)
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

    if (warp == 0 && lane == 0) {
        // ---- producer: the W box (128 features x 64 inputs) and the x box (BN tokens x 64 inputs)
        const uint64_t pol_w = l2_policy_evict_first();  // each weight tile is read by one CTA per token tile
        const uint64_t pol_x = l2_policy_evict_last();   // x is read by every output tile
        for (int k = k0; k < k1; ++k) {
            const int i = k - k0, st = i % S::kStages;
            if (i >= S::kStages && !mbar_wait(bar_empty + 8 * st, ((i / S::kStages) - 1) & 1)) {
                atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            const uint32_t a = base + st * S::kStageBytes, fb = bar_full + 8 * st;
            mbar_arrive_expect_tx(fb, S::kStageBytes);
            tma_load_2d(a, &tmW, k * kBK, m0, fb, pol_w);
            tma_load_2d(a + S::kABytes, &tmX, k * kBK, n0, fb, pol_x);
        }
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
    const bool ok = mbar_wait(bar_done, 0);
    tc_fence_after();
    const int o = m0 + 32 * warp + lane;
    if (ok && k1 > k0) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
            tmem_wait_ld_regs(v);
            if (p.splits == 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = n0 + c0 + j;
                    if (t < p.tokens) p.y[(int64_t)t * p.out + o] = __float2bfloat16_rn(__uint_as_float(v[j]));
                }
            } else {
                float* dst = p.part + (int64_t)split * p.tokens * p.out;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = n0 + c0 + j;
                    if (t < p.tokens) dst[(int64_t)t * p.out + o] = __uint_as_float(v[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, BN);
    }
}

// y = bf16 of the sum of the split partials, in split order.
__global__ void __launch_bounds__(256) linear_reduce_kernel(LinParams p)
{
    const int64_t n4 = (int64_t)p.tokens * p.out / 4;
    const int64_t stride = (int64_t)p.tokens * p.out / 4;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 acc = reinterpret_cast<const float4*>(p.part)[i];
        for (int s = 1; s < p.splits; ++s) {
            const float4 b = reinterpret_cast<const float4*>(p.part)[s * stride + i];
            acc.x += b.x;
            acc.y += b.y;
            acc.z += b.z;
            acc.w += b.w;
        }
        uint2 r;
        r.x = pack_bf16(__float2bfloat16_rn(acc.x), __float2bfloat16_rn(acc.y));
        r.y = pack_bf16(__float2bfloat16_rn(acc.z), __float2bfloat16_rn(acc.w));
        reinterpret_cast<uint2*>(p.y)[i] = r;
    }
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
    const dim3 grid(p.out / kBM, (p.tokens + BN - 1) / BN, splits);
    const bool timed = pool->timer_on;
    const int slot = (int)(pool->timer_count % kTimerSlots);
    if (timed && (e = cudaEventRecord(pool->ev_start[slot], s)) != cudaSuccess) return e;
    linear_kernel<BN><<<grid, kLinThreads, S::kAlloc, s>>>(tmW, tmX, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (timed) {
        if ((e = cudaEventRecord(pool->ev_stop[slot], s)) != cudaSuccess) return e;
        pool->timer_count++;
    }
    if (splits == 1) return cudaSuccess;
    const int64_t n4 = (int64_t)p.tokens * p.out / 4;
    const int blocks = (int)((n4 + 255) / 256 < 4 * pool->num_sms ? (n4 + 255) / 256 : 4 * pool->num_sms);
    linear_reduce_kernel<<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int linear_tile_tokens(int tokens) { return tokens <= 64 ? 64 : tokens <= 128 ? 128 : 256; }

// Split the input features over CTAs only while the output tiles alone fill
// less than half the SMs, and keep at least 4 steps of 64 per split.
int linear_splits(const pkv_pool* pool, int tokens, int in, int out)
{
    const int bn = linear_tile_tokens(tokens);
    const int tiles = (out / kBM) * ((tokens + bn - 1) / bn);
    int splits = 1;
    while (tiles * splits * 2 <= pool->num_sms && (in / kBK) / (splits * 2) >= 4) splits *= 2;
    return splits;
}

cudaError_t launch_linear(pkv_pool* pool, const void* x, const void* w, void* y, int tokens, int in, int out,
                          void* part, cudaStream_t s)
{
    LinParams p;
    p.y = static_cast<__nv_bfloat16*>(y);
    p.part = static_cast<float*>(part);
    p.err = pool->err;
    p.tokens = tokens;
    p.in = in;
    p.out = out;
    p.splits = linear_splits(pool, tokens, in, out);
    switch (linear_tile_tokens(tokens)) {
    case 64:
        return launch_linear_bn<64>(pool, x, w, p, p.splits, s);
    case 128:
        return launch_linear_bn<128>(pool, x, w, p, p.splits, s);
    default:
        return launch_linear_bn<256>(pool, x, w, p, p.splits, s);
    }
}

}  // namespace pkv
