// Device-side building blocks shared by the kernels of the sharded
// mixed-precision FlatParameter step (reduce-scatter by averaging, AdamW on
// each rank's fp32 shard, bf16 cast, all-gather).
//
// Data layout in HBM (all buffers caller-owned):
//   grads[k]      bf16, P_pad elements: logical rank k's full flat gradient
//   master/m/v[r] fp32, S elements: rank r's shard of the optimizer state
//   accum[r]      fp32, S elements: rank r's micro-step accumulator
//   out[o]        bf16, P_pad elements: the all-gathered parameters
// Rank r's shard covers flat elements [r*S, (r+1)*S).  Shard-local buffers
// start 16-byte aligned, so an 8-element group at a shard-local index that is
// a multiple of 8 is two aligned 16-byte fp32 vectors.  Flat buffers are
// indexed at r*S + j, which is aligned only when r*S is a multiple of 8;
// otherwise the gradient loads are realigned in registers (align_shift) and
// the parameter stores are narrowed (store_bf16x8).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace zf {

constexpr int kVec = 8;                 // elements per thread per group (16 B of bf16)
constexpr int kThreads = 256;           // threads per CTA
constexpr int kTile = kThreads * kVec;  // shard elements per CTA tile

// Optimizer constants derived on the host in double precision and rounded
// once to fp32.
// The moment coefficients are carried as (hi, lo) fp32 pairs, hi + lo being
// the double-precision value to ~2^-48: with a single fp32 constant
// (0.9f = 0.89999998) the moment recursions would pick up a bias of ~3e-8
// relative per step that accumulates coherently over the steps.
struct AdamConsts {
    float beta1, beta1_lo, one_minus_beta1, one_minus_beta1_lo;
    float beta2, beta2_lo, one_minus_beta2, one_minus_beta2_lo;
    float eps;
    float lr_wd;         // lr * weight_decay (decoupled decay theta -= lr*wd*theta)
    float step_size;     // lr / (1 - beta1^t)
    float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
    float divisor;       // micro-steps averaged (1 for a plain step)
};

// ---------------------------------------------------------------- bf16 ----

// Two bf16 in one 32-bit word (lower index in the low half) -> two fp32.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float bf16_to_float(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_rn(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(float_to_bf16_rn(lo)) |
           (static_cast<uint32_t>(float_to_bf16_rn(hi)) << 16);
}

// ------------------------------------------------- compensated summation ----
//
// Knuth's error-free two-sum: after t = s + x, (s - (t - (t - s))) + (x - (t - s))
// is exactly the rounding error of t.  The errors are collected in c, so that
// s + c carries the running sum of the ranks' gradients to about twice fp32
// precision.  Packed over element pairs with the sm_100+ f32x2 additions
// (FADD2), written in PTX on 64-bit register pairs from end to end: as C++ on
// float2 values (a - b as an fma with a (-1, -1) pair) the compiler spent
// about five register moves per two-sum forming pairs, and the clipped step's
// norm pass, bound by instruction issue, ran 7 % more instructions and 1.4 %
// slower.  The scalar form below performs the identical IEEE operations lane
// by lane, so the packed and scalar paths give bit-identical sums.

__device__ __forceinline__ void two_sum_add2(float2& s, float2& c, float2 x) {
    asm("{\n\t.reg .b64 xp, sp, cp, t, bp, ap, db, da, e;\n\t"
        "mov.b64 xp, {%4, %5};\n\t"
        "mov.b64 sp, {%0, %1};\n\t"
        "mov.b64 cp, {%2, %3};\n\t"
        "add.rn.f32x2 t, sp, xp;\n\t"
        "sub.rn.f32x2 bp, t, sp;\n\t"
        "sub.rn.f32x2 ap, t, bp;\n\t"
        "sub.rn.f32x2 db, xp, bp;\n\t"
        "sub.rn.f32x2 da, sp, ap;\n\t"
        "add.rn.f32x2 e, da, db;\n\t"
        "add.rn.f32x2 cp, cp, e;\n\t"
        "mov.b64 {%0, %1}, t;\n\t"
        "mov.b64 {%2, %3}, cp;\n\t}"
        : "+f"(s.x), "+f"(s.y), "+f"(c.x), "+f"(c.y)
        : "f"(x.x), "f"(x.y));
}

// The same for two bf16 gradient values in one 32-bit word (lower index in the
// low half), widened to fp32 inside the same PTX block.
__device__ __forceinline__ void two_sum_add_bf16x2(float2& s, float2& c, uint32_t w) {
    asm("{\n\t.reg .b32 xl, xh;\n\t.reg .b64 xp, sp, cp, t, bp, ap, db, da, e;\n\t"
        "shl.b32 xl, %4, 16;\n\t"
        "and.b32 xh, %4, 0xFFFF0000;\n\t"
        "mov.b64 xp, {xl, xh};\n\t"
        "mov.b64 sp, {%0, %1};\n\t"
        "mov.b64 cp, {%2, %3};\n\t"
        "add.rn.f32x2 t, sp, xp;\n\t"
        "sub.rn.f32x2 bp, t, sp;\n\t"
        "sub.rn.f32x2 ap, t, bp;\n\t"
        "sub.rn.f32x2 db, xp, bp;\n\t"
        "sub.rn.f32x2 da, sp, ap;\n\t"
        "add.rn.f32x2 e, da, db;\n\t"
        "add.rn.f32x2 cp, cp, e;\n\t"
        "mov.b64 {%0, %1}, t;\n\t"
        "mov.b64 {%2, %3}, cp;\n\t}"
        : "+f"(s.x), "+f"(s.y), "+f"(c.x), "+f"(c.y)
        : "r"(w));
}

__device__ __forceinline__ float sub1(float a, float b) { return __fmaf_rn(b, -1.0f, a); }

__device__ __forceinline__ void two_sum_add1(float& s, float& c, float x) {
    const float t = __fadd_rn(s, x);
    const float bp = sub1(t, s);
    const float ap = sub1(t, bp);
    const float db = sub1(x, bp);
    const float da = sub1(s, ap);
    c = __fadd_rn(c, __fadd_rn(da, db));
    s = t;
}

// Mean over n ranks from the compensated pair (s, c).  For a power-of-two n
// the scaling is exact, so the mean is RN(s + c) * (1/n).  Otherwise the
// quotient q = RN(s/n) is corrected by the exact remainder s - q*n (one fma)
// and the error term c, which keeps the result correctly rounded in almost
// every case instead of rounding twice.
__device__ __forceinline__ float finish_mean(float s, float c, float n_f, float inv_n, bool pow2) {
    if (pow2) return __fmul_rn(__fadd_rn(s, c), inv_n);
    const float q = __fdiv_rn(s, n_f);
    const float r = __fmaf_rn(-q, n_f, s);
    return __fadd_rn(q, __fdiv_rn(__fadd_rn(r, c), n_f));
}

// The first rank's values start the sum: s = x + 0 and c = s - s are exactly
// what a two-sum of x into (0, 0) leaves (+0 for a -0 input, +0 error terms
// for finite values, NaN error terms for infinities and NaNs), in two packed
// additions instead of seven.
__device__ __forceinline__ void first_rank2(float2& s, float2& c, float2 x) {
    asm("{\n\t.reg .b64 xp, zp, t, e;\n\t"
        "mov.b64 xp, {%4, %5};\n\t"
        "mov.b64 zp, 0;\n\t"
        "add.rn.f32x2 t, zp, xp;\n\t"
        "sub.rn.f32x2 e, t, t;\n\t"
        "mov.b64 {%0, %1}, t;\n\t"
        "mov.b64 {%2, %3}, e;\n\t}"
        : "=f"(s.x), "=f"(s.y), "=f"(c.x), "=f"(c.y)
        : "f"(x.x), "f"(x.y));
}

// The same for two bf16 values in one word, widened inside the PTX block.
__device__ __forceinline__ void first_rank_bf16x2(float2& s, float2& c, uint32_t w) {
    asm("{\n\t.reg .b32 xl, xh;\n\t.reg .b64 xp, zp, t, e;\n\t"
        "shl.b32 xl, %4, 16;\n\t"
        "and.b32 xh, %4, 0xFFFF0000;\n\t"
        "mov.b64 xp, {xl, xh};\n\t"
        "mov.b64 zp, 0;\n\t"
        "add.rn.f32x2 t, zp, xp;\n\t"
        "sub.rn.f32x2 e, t, t;\n\t"
        "mov.b64 {%0, %1}, t;\n\t"
        "mov.b64 {%2, %3}, e;\n\t}"
        : "=f"(s.x), "=f"(s.y), "=f"(c.x), "=f"(c.y)
        : "r"(w));
}

__device__ __forceinline__ void first_rank_bf16x8(float2 (&s)[4], float2 (&c)[4], uint4 w) {
    first_rank_bf16x2(s[0], c[0], w.x);
    first_rank_bf16x2(s[1], c[1], w.y);
    first_rank_bf16x2(s[2], c[2], w.z);
    first_rank_bf16x2(s[3], c[3], w.w);
}

// Accumulate one rank's 8 bf16 gradient values (a 16-byte word group).
__device__ __forceinline__ void two_sum_add_bf16x8(float2 (&s)[4], float2 (&c)[4], uint4 w) {
    two_sum_add_bf16x2(s[0], c[0], w.x);
    two_sum_add_bf16x2(s[1], c[1], w.y);
    two_sum_add_bf16x2(s[2], c[2], w.z);
    two_sum_add_bf16x2(s[3], c[3], w.w);
}

// The same two-sums written as C++ on float2 values (a - b as an fma with a
// (-1, -1) pair): the same IEEE operations, so the same bits.  The direct-load
// kernels use this form: they hold many loads in registers, and with the PTX
// blocks ptxas spilled in them (up to 68 bytes).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}

__device__ __forceinline__ void two_sum_add2_c(float2& s, float2& c, float2 x) {
    const float2 t = __fadd2_rn(s, x);
    const float2 bp = sub2(t, s);
    const float2 ap = sub2(t, bp);
    const float2 db = sub2(x, bp);
    const float2 da = sub2(s, ap);
    c = __fadd2_rn(c, __fadd2_rn(da, db));
    s = t;
}

__device__ __forceinline__ void two_sum_add_bf16x8_c(float2 (&s)[4], float2 (&c)[4], uint4 w) {
    two_sum_add2_c(s[0], c[0], bf16x2_to_float2(w.x));
    two_sum_add2_c(s[1], c[1], bf16x2_to_float2(w.y));
    two_sum_add2_c(s[2], c[2], bf16x2_to_float2(w.z));
    two_sum_add2_c(s[3], c[3], bf16x2_to_float2(w.w));
}

// ------------------------------------------------------------- loads -------

// Read-once streams: cache-streaming loads (evict-first).
__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void ld_f32x8(const float* p, float (&x)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void st_f32x8(float* p, const float (&x)[8]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
    __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(x[4], x[5], x[6], x[7]));
}

// Eight bf16 starting A elements into the 16 aligned elements w0:w1.
template <int A>
__device__ __forceinline__ uint4 align_shift(uint4 w0, uint4 w1) {
    if constexpr (A == 0) {
        return w0;
    } else {
        const uint32_t W[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        constexpr int q = A / 2;
        uint4 r;
        if constexpr (A % 2 == 0) {
            r.x = W[q];
            r.y = W[q + 1];
            r.z = W[q + 2];
            r.w = W[q + 3];
        } else {
            // high half of word q+i and low half of word q+i+1
            r.x = __byte_perm(W[q], W[q + 1], 0x5432);
            r.y = __byte_perm(W[q + 1], W[q + 2], 0x5432);
            r.z = __byte_perm(W[q + 2], W[q + 3], 0x5432);
            r.w = __byte_perm(W[q + 3], W[q + 4], 0x5432);
        }
        return r;
    }
}

// Store 8 packed bf16 (4 words) at flat element index e of a bf16 buffer
// whose base is 16-byte aligned; `mis` = e mod 8 selects the widest legal
// store.
__device__ __forceinline__ void store_bf16x8(uint16_t* base, int64_t e, int mis, uint4 w) {
    if (mis == 0) {
        *reinterpret_cast<uint4*>(base + e) = w;
    } else if ((mis & 3) == 0) {
        uint2* p = reinterpret_cast<uint2*>(base + e);
        p[0] = make_uint2(w.x, w.y);
        p[1] = make_uint2(w.z, w.w);
    } else if ((mis & 1) == 0) {
        uint32_t* p = reinterpret_cast<uint32_t*>(base + e);
        p[0] = w.x;
        p[1] = w.y;
        p[2] = w.z;
        p[3] = w.w;
    } else {
        uint16_t* p = base + e;
        p[0] = static_cast<uint16_t>(w.x);
        p[1] = static_cast<uint16_t>(w.x >> 16);
        p[2] = static_cast<uint16_t>(w.y);
        p[3] = static_cast<uint16_t>(w.y >> 16);
        p[4] = static_cast<uint16_t>(w.z);
        p[5] = static_cast<uint16_t>(w.z >> 16);
        p[6] = static_cast<uint16_t>(w.w);
        p[7] = static_cast<uint16_t>(w.w >> 16);
    }
}

// Store 8 packed bf16 per lane for a whole warp whose lanes own consecutive
// 8-element groups starting at flat index e (lane 0) -- e, e+8, ... -- with
// e mod 8 = mis for every lane.  When mis != 0 the lanes' groups straddle the
// 16-byte grid: lane l builds the aligned block that holds its last mis
// elements and lane l+1's first 8-mis (one shuffle per word), so lanes 0..30
// each issue one aligned 16-byte store; lane 0's leading and lane 31's
// trailing partial blocks are written element by element.  Every lane of the
// warp must call this (the shuffles use the full mask).
template <int MIS>
__device__ __forceinline__ void store_bf16x8_warp_mis(uint16_t* base, int64_t e, uint4 w,
                                                      int lane) {
    uint4 nx;
    nx.x = __shfl_down_sync(0xFFFFFFFFu, w.x, 1);
    nx.y = __shfl_down_sync(0xFFFFFFFFu, w.y, 1);
    nx.z = __shfl_down_sync(0xFFFFFFFFu, w.z, 1);
    nx.w = __shfl_down_sync(0xFFFFFFFFu, w.w, 1);
    const uint4 blk = align_shift<8 - MIS>(w, nx);
    if (lane < 31) *reinterpret_cast<uint4*>(base + e - MIS + 8) = blk;
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < 8 - MIS; ++t) {
            base[e + t] = static_cast<uint16_t>(words[t >> 1] >> ((t & 1) * 16));
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int t = 8 - MIS; t < 8; ++t) {
            base[e + t] = static_cast<uint16_t>(words[t >> 1] >> ((t & 1) * 16));
        }
    }
}

__device__ __forceinline__ void store_bf16x8_warp(uint16_t* base, int64_t e, int mis, uint4 w,
                                                  int lane) {
    switch (mis) {
        case 0: *reinterpret_cast<uint4*>(base + e) = w; break;
        case 1: store_bf16x8_warp_mis<1>(base, e, w, lane); break;
        case 2: store_bf16x8_warp_mis<2>(base, e, w, lane); break;
        case 3: store_bf16x8_warp_mis<3>(base, e, w, lane); break;
        case 4: store_bf16x8_warp_mis<4>(base, e, w, lane); break;
        case 5: store_bf16x8_warp_mis<5>(base, e, w, lane); break;
        case 6: store_bf16x8_warp_mis<6>(base, e, w, lane); break;
        default: store_bf16x8_warp_mis<7>(base, e, w, lane); break;
    }
}

// ------------------------------------------------------------- AdamW -------
//
// One element of the local shard update: decoupled weight decay, the two
// moments, bias-corrected step, all in fp32 with explicit round-to-nearest
// intrinsics (no contraction decided by the compiler), IEEE sqrt and divide:
//   m' = beta1*m + (1-beta1)*g          v' = beta2*v + (1-beta2)*g^2
//   theta' = theta - lr*wd*theta - (lr/bc1) * m' / (sqrt(v')/sqrt(bc2) + eps)
__device__ __forceinline__ void adamw_update(const AdamConsts& k, float g, float& theta,
                                             float& m, float& v) {
    const float corr_m = __fmaf_rn(k.beta1_lo, m, __fmul_rn(k.one_minus_beta1_lo, g));
    const float m_new = __fmaf_rn(k.beta1, m, __fmaf_rn(k.one_minus_beta1, g, corr_m));
    const float gg = __fmul_rn(g, g);
    const float corr_v = __fmaf_rn(k.beta2_lo, v, __fmul_rn(k.one_minus_beta2_lo, gg));
    const float v_new = __fmaf_rn(k.beta2, v, __fmaf_rn(k.one_minus_beta2, gg, corr_v));
    const float denom = __fmaf_rn(__fsqrt_rn(v_new), k.inv_sqrt_bc2, k.eps);
    const float upd = __fdiv_rn(m_new, denom);
    const float decayed = __fmaf_rn(-k.lr_wd, theta, theta);
    theta = __fmaf_rn(-k.step_size, upd, decayed);
    m = m_new;
    v = v_new;
}

// Two elements at once: the operations of adamw_update, lane by lane, on
// packed fp32 pairs.  FFMA2 / FMUL2 round each lane exactly as the scalar
// instructions do, so the results are bit-identical to two adamw_update calls
// in fewer instructions (square root and division stay scalar).
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }

__device__ __forceinline__ void adamw_update2(const AdamConsts& k, float2 g, float2& theta,
                                              float2& m, float2& v) {
    const float2 corr_m =
        __ffma2_rn(splat2(k.beta1_lo), m, __fmul2_rn(splat2(k.one_minus_beta1_lo), g));
    const float2 m_new = __ffma2_rn(splat2(k.beta1), m,
                                    __ffma2_rn(splat2(k.one_minus_beta1), g, corr_m));
    const float2 gg = __fmul2_rn(g, g);
    const float2 corr_v =
        __ffma2_rn(splat2(k.beta2_lo), v, __fmul2_rn(splat2(k.one_minus_beta2_lo), gg));
    const float2 v_new = __ffma2_rn(splat2(k.beta2), v,
                                    __ffma2_rn(splat2(k.one_minus_beta2), gg, corr_v));
    const float2 root = make_float2(__fsqrt_rn(v_new.x), __fsqrt_rn(v_new.y));
    const float2 denom = __ffma2_rn(root, splat2(k.inv_sqrt_bc2), splat2(k.eps));
    const float2 upd = make_float2(__fdiv_rn(m_new.x, denom.x), __fdiv_rn(m_new.y, denom.y));
    const float2 decayed = __ffma2_rn(splat2(-k.lr_wd), theta, theta);
    theta = __ffma2_rn(splat2(-k.step_size), upd, decayed);
    m = m_new;
    v = v_new;
}

}  // namespace zf
