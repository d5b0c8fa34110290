// QK-norm and rotate-half RoPE of one head held by a warp, 4 consecutive dims
// per lane (lane l: dims 4l..4l+3): the per-token work before attention, shared
// by the attention kernels and the projection epilogue that can do it instead.
//
// qwen3-8b Nest files, src/norm.linnet (RmsNorm: x / sqrt(mean(x^2) + eps) * w)
// and src/rope.linnet (tables: angle pos * theta^(-2i/d), rotate-half pairing
// (i, i + d/2)); fantasma model.zig, applyRope (a partial rotation of the
// first rotary_dim dims).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ void unpack4(uint2 r, float (&x)[4])
{
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xffff0000u);
}

__device__ __forceinline__ uint2 pack4(const float (&y)[4])
{
    uint2 r;
    r.x = pack_bf16(__float2bfloat16_rn(y[0]), __float2bfloat16_rn(y[1]));
    r.y = pack_bf16(__float2bfloat16_rn(y[2]), __float2bfloat16_rn(y[3]));
    return r;
}

// 1 / sqrt(mean(x^2) + eps) over the warp's head (4 dims a lane), every
// operation spelled out, so that each kernel that inlines it gets the same bits
// (a plain a*b + c may be contracted to a fused multiply-add in one context and
// not in another).
__device__ __forceinline__ float inv_rms(const float (&x)[4], float eps)
{
    float ss = __fmaf_rn(x[3], x[3], __fmaf_rn(x[2], x[2], __fmaf_rn(x[1], x[1], __fmul_rn(x[0], x[0]))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, o));
    return rsqrtf(__fmaf_rn(ss, 1.0f / kHeadDim, eps));
}

// k after QK-norm + rotate-half RoPE, for the warp that holds one k head
// (lane l: elements 4l..4l+3; the rotate-half partner of element i < 64 is
// i + 64, in lane l ^ 16):
//   RMSNorm: x / sqrt(mean(x^2) + eps) * w;  RoPE: y*cos + rotate_half(y)*sin.
// Both are linear in y, so the normaliser goes last:
//   r = inv * a,  a = u*cos -/+ u'*sin,  u = x*w (exact in fp32: bf16 x bf16).
// k is stored in bf16, and when the two terms of a cancel, plain fp32 loses
// far more than a bf16 ulp.  So a is formed without error growth: cos and sin
// come as fp32 hi + lo pairs of the double values, the products' rounding
// errors are recovered exactly with fma and the sum's with two-sum; the
// result has fp32 accuracy relative to a itself, and rounds to within one
// bf16 ulp of the exact value.
__device__ __forceinline__ float rotate_exact(float u, float up, float2 hi, float2 lo)
{
    const float p1 = __fmul_rn(u, hi.x), e1 = __fmaf_rn(u, hi.x, -p1);
    const float p2 = __fmul_rn(up, hi.y), e2 = __fmaf_rn(up, hi.y, -p2);
    const float s = __fadd_rn(p1, p2);
    const float bp = __fsub_rn(s, p1);
    const float e3 = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, bp)), __fsub_rn(p2, bp));
    const float lo_terms = __fmaf_rn(u, lo.x, __fmaf_rn(up, lo.y, __fadd_rn(__fadd_rn(e1, e2), e3)));
    return __fadd_rn(s, lo_terms);
}

// RoPE layout of a warp holding one head, 4 consecutive dims per lane: with R
// rotated dims, lanes below R/8 hold the first rotary half (partner: R/2
// dims, i.e. R/8 lanes, up), lanes in [R/8, R/4) the second (partner R/8 lanes
// down), and lanes from R/4 up the dims RoPE leaves as they are.
struct KRope {
    int src;     // lane holding this lane's partner dims
    float sgn;   // -1: first half (u cos - partner sin), +1: second (u cos + partner sin)
    int f0;      // table index of this lane's first dim
    bool rot;    // false: not rotated
};
__device__ __forceinline__ KRope krope(int lane, int rot)
{
    const int hl = rot / 8;
    KRope r;
    r.rot = lane < 2 * hl;
    const bool first = lane < hl;
    r.src = first ? lane + hl : (r.rot ? lane - hl : lane);
    r.sgn = first ? -1.f : 1.f;
    r.f0 = r.rot ? 4 * (first ? lane : lane - hl) : 0;
    return r;
}

// The warp's normed + roped k as 4 bf16 (this lane's elements).
//   kraw: this lane's 4 raw bf16;  wk: its k_norm weights;
//   rh/rl: (cos, sin) hi and lo parts at the token's position for this lane's
//   table entries krope(lane, rot).f0 .. + 3;  rot: the rotated dims.
__device__ __forceinline__ uint2 norm_rope_k_regs(uint2 kraw, const float (&wk)[4], const float2 (&rh)[4],
                                                  const float2 (&rl)[4], float eps, int lane, int rot)
{
    float x[4];
    unpack4(kraw, x);
    const float inv = inv_rms(x, eps);
    const KRope kr = krope(lane, rot);
    __nv_bfloat16 r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float u = x[i] * wk[i];
        const float partner = kr.sgn * __shfl_sync(kFull, u, kr.src);
        r[i] = __float2bfloat16_rn(__fmul_rn(kr.rot ? rotate_exact(u, partner, rh[i], rl[i]) : u, inv));
    }
    return make_uint2(pack_bf16(r[0], r[1]), pack_bf16(r[2], r[3]));
}

//   rhi/rlo: (cos, sin) hi and lo parts of the token's position, [64].
__device__ __forceinline__ uint2 norm_rope_k(uint2 kraw, const float (&wk)[4], const float2* rhi, const float2* rlo,
                                             float eps, int lane, int rot)
{
    const KRope kr = krope(lane, rot);
    float2 rh[4], rl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        rh[i] = rhi[kr.f0 + i];
        rl[i] = rlo[kr.f0 + i];
    }
    return norm_rope_k_regs(kraw, wk, rh, rl, eps, lane, rot);
}

// The warp's normed + roped q in fp32 (this lane's 4 dims), rotated with the
// fp32 nearest (cos, sin) rh of each of its table entries.  The attention
// splits q into a bf16 head and remainder afterwards, so fp32 is enough here.
__device__ __forceinline__ float4 norm_rope_q_regs(uint2 qraw, const float (&wq)[4], const float2 (&rh)[4], float eps,
                                                   int lane, int rot)
{
    float x[4];
    unpack4(qraw, x);
    const float inv = inv_rms(x, eps);
    const KRope kr = krope(lane, rot);
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float u = x[i] * wq[i];
        const float partner = kr.sgn * __shfl_sync(kFull, u, kr.src);
        y[i] = inv * (kr.rot ? u * rh[i].x + partner * rh[i].y : u);
    }
    return make_float4(y[0], y[1], y[2], y[3]);
}

}  // namespace pkv
