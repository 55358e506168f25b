// device_common.cuh - device helpers shared by the backward and forward
// kernels: mbarrier and bulk-copy PTX wrappers with bounded waits, packed
// fp32x2 arithmetic, 16-bit packing, and the row cursor of a CTA range.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mcc1d {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete; gives up
// (returns false) after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded_inline(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// The same, out of line (keeps the slow path out of the hot loops). Kernels
// that split their registers by warpgroup (setmaxnreg) take the inline form:
// one out-of-line body cannot serve regions of different register counts.
static __device__ __noinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    return mbar_wait_bounded_inline(bar, parity);
}

// Global -> shared bulk copy completing on an mbarrier (no multicast).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Shared -> global bulk copy of one row, in the issuing thread's bulk-async
// group (16-byte aligned addresses, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Every committed group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group of this thread has completed (its writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Packed fp32x2 arithmetic (sm_100+), each lane rounded to nearest even.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// ------------------------------------------------------------------ 16-bit types
// DT 0 = bf16, 1 = fp16. A consumer thread owns 2*NP channels: NP = 4 moves
// 16 bytes per row (uint4), NP = 2 moves 8 bytes (uint2).
template <int NP>
struct Vf {
    float2 e[NP];
};

template <int NP>
struct Raw {
    uint32_t u[NP];
};

template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t u)
{
    if (DT == 0) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    } else {
        union {
            uint32_t u;
            __half2 h;
        } c;
        c.u = u;
        return __half22float2(c.h);
    }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float2 v)
{
    if (DT == 0) {
        union {
            __nv_bfloat162 b;
            uint32_t u;
        } c;
        c.b = __floats2bfloat162_rn(v.x, v.y);
        return c.u;
    } else {
        union {
            __half2 h;
            uint32_t u;
        } c;
        c.h = __floats2half2_rn(v.x, v.y);
        return c.u;
    }
}

// Plain vector load (shared or global memory).
template <int NP>
__device__ __forceinline__ Raw<NP> load_raw(const void *p)
{
    Raw<NP> r;
    if constexpr (NP == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        r.u[0] = v.x;
        r.u[1] = v.y;
        r.u[2] = v.z;
        r.u[3] = v.w;
    } else {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        r.u[0] = v.x;
        r.u[1] = v.y;
    }
    return r;
}

// Read-only global load through the non-coherent path.
template <int NP>
__device__ __forceinline__ Raw<NP> ldg_raw(const void *p)
{
    Raw<NP> r;
    if constexpr (NP == 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        r.u[0] = v.x;
        r.u[1] = v.y;
        r.u[2] = v.z;
        r.u[3] = v.w;
    } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        r.u[0] = v.x;
        r.u[1] = v.y;
    }
    return r;
}

// Streaming (evict-first) global store.
template <int NP>
__device__ __forceinline__ void store_cs(void *p, const uint32_t (&u)[NP])
{
    if constexpr (NP == 4)
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(u[0], u[1], u[2], u[3]));
    else
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(u[0], u[1]));
}

template <int DT, int NP>
__device__ __forceinline__ Vf<NP> unpack(const Raw<NP> &r)
{
    Vf<NP> v;
#pragma unroll
    for (int e = 0; e < NP; ++e)
        v.e[e] = unpack2<DT>(r.u[e]);
    return v;
}

// A staged gradY row, masked by clearing the bits (exact +0 whatever the
// staged bytes hold; rows past the end of S carry a zero mask byte).
template <int DT, int NP>
__device__ __forceinline__ Vf<NP> load_masked(const uint8_t *p, uint8_t keep_byte)
{
    Raw<NP> r = load_raw<NP>(p);
    const uint32_t keep = 0u - (uint32_t)keep_byte;
#pragma unroll
    for (int e = 0; e < NP; ++e)
        r.u[e] &= keep;
    return unpack<DT, NP>(r);
}

// One channel pair (4 bytes) of a staged row, masked like load_masked.
template <int DT>
__device__ __forceinline__ float2 load_masked_pair(const uint8_t *p, uint8_t keep_byte)
{
    return unpack2<DT>(*reinterpret_cast<const uint32_t *>(p) & (0u - (uint32_t)keep_byte));
}

// Channel pair e of v, e a run-time index (selects, no local memory).
template <int NP>
__device__ __forceinline__ float2 pick_pair(const Vf<NP> &v, int e)
{
    float2 r = v.e[0];
#pragma unroll
    for (int t = 1; t < NP; ++t)
        if (e == t)
            r = v.e[t];
    return r;
}

// ------------------------------------------------------------------ sums of W products
// The gradX (and forward y) value of a channel is a sum of W products of two
// 16-bit values. Each product is exact in fp32 (8 x 8 or 11 x 11 significant
// bits), so only the additions round. A TwoSum cascade over the first W-1
// products keeps every rounding error, the last product is added plainly,
// then the summed errors: within a hair of the exact sum, rounded once to
// the 16-bit type (W = 3: TwoSum of the first two, one more add, the
// correction). prod(k) returns product k for two channels.
template <int DT, int W, typename Prod>
__device__ __forceinline__ uint32_t sum_to16(Prod prod)
{
    float2 pk[W];
#pragma unroll
    for (int k = 0; k < W; ++k)
        pk[k] = prod(k);
    float2 s = pk[0], err = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 1; k < W - 1; ++k) {
        const float2 sn = add2(s, pk[k]);
        const float2 bb = sub2(sn, s);
        const float2 ek = add2(sub2(s, sub2(sn, bb)), sub2(pk[k], bb));
        err = (k == 1) ? ek : add2(err, ek);
        s = sn;
    }
    if constexpr (W >= 3)
        return pack2<DT>(add2(add2(s, pk[W - 1]), err));
    else if constexpr (W == 2)
        return pack2<DT>(add2(s, pk[1]));
    else
        return pack2<DT>(s);
}

// s = sum_k a(k) b(k) for W <= 8 in a fixed tree of depth <= 3: each pair
// a(2j) b(2j) + a(2j+1) b(2j+1) by one multiply and one fused multiply-add
// (products of two 16-bit values are exact in fp32, so a pair rounds once),
// then the pairs' tree; an odd last product is fused into the last pair.
template <int W, typename A, typename B>
__device__ __forceinline__ float2 dot_tree(A a, B b)
{
    static_assert(W >= 1 && W <= 8, "the depth-3 tree holds up to 8 products");
    if constexpr (W == 1) {
        return mul2(a(0), b(0));
    } else {
        constexpr int kPairs = W / 2;
        float2 pr[kPairs];
#pragma unroll
        for (int j = 0; j < kPairs; ++j)
            pr[j] = fma2(a(2 * j + 1), b(2 * j + 1), mul2(a(2 * j), b(2 * j)));
        if constexpr (W & 1)
            pr[kPairs - 1] = fma2(a(W - 1), b(W - 1), pr[kPairs - 1]);
        if constexpr (kPairs == 1)
            return pr[0];
        else if constexpr (kPairs == 2)
            return add2(pr[0], pr[1]);
        else if constexpr (kPairs == 3)
            return add2(add2(pr[0], pr[1]), pr[2]);
        else
            return add2(add2(pr[0], pr[1]), add2(pr[2], pr[3]));
    }
}

// Upper bounds, per lane, by rounding toward +infinity: s + |v|, s - |v|,
// a * b.
__device__ __forceinline__ float2 add_abs_ru(float2 s, float2 v)
{
    return make_float2(__fadd_ru(s.x, fabsf(v.x)), __fadd_ru(s.y, fabsf(v.y)));
}
__device__ __forceinline__ float2 sub_abs_ru(float2 s, float2 v)
{
    return make_float2(__fsub_ru(s.x, fabsf(v.x)), __fsub_ru(s.y, fabsf(v.y)));
}
__device__ __forceinline__ float2 mul_ru(float2 a, float2 b)
{
    return make_float2(__fmul_ru(a.x, b.x), __fmul_ru(a.y, b.y));
}

// Where the certified sum replaces the cascade (both dtypes), measured
// against it kernel by kernel: the backward from W = 5 (at W = 4 the
// cascade, in its two-CTA kernel, was faster: 0.83 of peak against 0.70),
// the forward from W = 4.
constexpr int kCertMinWBwd = 5;
constexpr int kCertMinWFwd = 4;

// Certificate for a sum s of W <= 8 exact products p_k = g_k w_k formed by
// dot_tree, a = sum_k |p_k|, u = 2^-24. Each addition's rounding error is
// at most u times its computed result (Higham, "Accuracy and Stability of
// Numerical Algorithms", 2nd ed., (2.5)), and s - exact is the sum of those
// errors. The nodes of one level of the tree below the root cover disjoint
// sets of products, so their magnitudes add up to at most a (1 + 2u): with
// L such levels (L = 1 up to W = 4: the pairs; L = 2 for W = 5..8: the
// pairs, then the pairs' pairs or an odd product fused into the last pair),
//     |s - exact| <= u (L a (1 + 2u) + |s|) =: E.
// The 16-bit grid's spacing at x exceeds x * 2^-(m+1) (m + 1 significant
// bits: 11 for fp16, 8 for bf16), so if E < (|s| - E) 2^-(m+1), s and the
// exact sum lie closer than the smallest spacing between them: at most one
// rounding boundary separates them and round(s) is within 1 ulp of the exact
// sum rounded once. Solved for |s| that is
//     |s| > L a u 2^(m+1) (1 + 2^-(m+1)) / (1 - u 2^(m+1) (1 + 2^-(m+1))) (1 + 2u),
// which cert_factor<DT, W>() * a covers (the last factor and the rounding of
// the constants within its (1 + 2^-20)). The kernels test
// cert_factor * max_k|w_k| * sum_k|g_k| <= |s|, whose left side, formed
// with upward rounding, is at least cert_factor * a.
template <int DT, int W>
__host__ __device__ constexpr float cert_factor()
{
    static_assert(W >= 1 && W <= 8, "dot_tree's levels are counted for W <= 8");
    constexpr float kL = W <= 4 ? 1.f : 2.f;
    // u 2^(m+1) = 2^-13 (fp16), 2^-16 (bf16); the quotient times (1 + 2^-20)
    // is 1.000611 (fp16) and 1.003923 (bf16), rounded up here
    return DT == 1 ? kL * 1.220703125e-4f * 1.00062f : kL * 1.52587890625e-5f * 1.00393f;
}

// ------------------------------------------------------------------ row cursor
// Position in the flattened (hb, j, i) row sequence of one CTA range.
struct Cursor {
    int64_t pos, end, i;
    int32_t j, hb;

    __device__ __forceinline__ void init(int64_t r0, int64_t r1, int64_t S, int64_t BS)
    {
        pos = r0;
        end = r1;
        hb = (int32_t)(r0 / BS);
        const int64_t rem = r0 - (int64_t)hb * BS;
        j = (int32_t)(rem / S);
        i = rem - (int64_t)j * S;
    }
    // Rows of the next stage: at most R, never across a sequence end or the range end.
    template <int R>
    __device__ __forceinline__ int rows(int64_t S) const
    {
        int64_t n = S - i;
        if (end - pos < n)
            n = end - pos;
        return n < R ? (int)n : R;
    }
    __device__ __forceinline__ void advance(int n, int64_t S, int32_t B)
    {
        pos += n;
        i += n;
        if (i == S) {
            i = 0;
            if (++j == B) {
                j = 0;
                ++hb;
            }
        }
    }
};

}  // namespace mcc1d
