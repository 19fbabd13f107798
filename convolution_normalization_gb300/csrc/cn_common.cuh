// Device helpers shared by the conv_norm kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <cuda.h>

#define CN_DEV __device__ __forceinline__
#define CN_PRAGMA(x) _Pragma(#x)
#define CN_UNROLL(n) CN_PRAGMA(unroll n)
// Unroll depth of the kernel-tap loops outside the innermost (kw, output)
// block.  1 keeps each loop body a few KB of code so it stays resident in
// the instruction cache; full unrolling repeats the FFMA block K^2 (or K^3)
// times and measured 1.4x slower on the 3-D mean kernel.
#ifndef CN_TAP_UNROLL
#define CN_TAP_UNROLL 1
#endif
// Unroll depth of the kh loop (the loop directly around one input-row load)
// of the 3-D mean kernel: 4 measured fastest (0.756 / 0.729 / 0.710 ms for
// 1 / 2 / 4 on the n512 workload).
#ifndef CN_KH_UNROLL
#define CN_KH_UNROLL 4
#endif

namespace cn {

// ---- activations -----------------------------------------------------------
enum { ACT_NONE = 0, ACT_HARDSWISH = 1, ACT_GELU = 2, ACT_SOFTMAX = 3 };

// HardSwish: v * clamp(v + 3, 0, 6) / 6  (l2_p27, HardSwish definition).
CN_DEV float hardswish(float v) {
    return v * fminf(fmaxf(v + 3.0f, 0.0f), 6.0f) * (1.0f / 6.0f);
}
// erf by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26 (Hastings' rational approximation): for x >= 0,
//   erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
//   t = 1 / (1 + p x),  |error| <= 1.5e-7;  erf(-x) = -erf(x).
// The constants, and the GELU below built from them, are checked against
// the stated bound by a CPU test.
#define CN_AS_P 0.3275911f
#define CN_AS_A1 0.254829592f
#define CN_AS_A2 -0.284496736f
#define CN_AS_A3 1.421413741f
#define CN_AS_A4 -1.453152027f
#define CN_AS_A5 1.061405429f
// Hardware approximations (PTX rcp.approx / ex2.approx, ~1 ulp).
CN_DEV float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
CN_DEV float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// Exact (erf-form) GELU: 0.5 v (1 + erf(v / sqrt 2))  (l2_p19, nn.GELU's
// default approximate='none'), with erf from 7.1.26 at x = |v| / sqrt 2.
// There 0.5 (1 - erf(x)) = g = 0.5 y(t) exp(-v^2 / 2) >= 0, so
//   GELU(v) = v - v g = max(v, 0) - |v| g   for v >= 0,
//   GELU(v) = v g     = max(v, 0) - |v| g   for v < 0,
// with 1/sqrt 2 folded into p, the 0.5 into the a_i and log2(e) / 2 into
// the exponent: 11 operations, one reciprocal and one exp2.
CN_DEV float gelu_erf(float v) {
    const float av = fabsf(v);
    const float t = rcp_approx(fmaf(CN_AS_P * 0.70710678118654752f, av, 1.0f));
    float y = fmaf(t, 0.5f * CN_AS_A5, 0.5f * CN_AS_A4);
    y = fmaf(t, y, 0.5f * CN_AS_A3);
    y = fmaf(t, y, 0.5f * CN_AS_A2);
    y = fmaf(t, y, 0.5f * CN_AS_A1);
    y *= t;
    const float e = ex2_approx(v * (v * (-0.5f * 1.4426950408889634f)));
    return fmaf(-av, y * e, fmaxf(v, 0.0f));
}
// ---- packed fp32 pairs (one instruction for two lanes of a float2) -----------
// Each lane is rounded as the scalar operation rounds it (round to nearest;
// fma fused), so pairs give the same bits as two scalar operations.
CN_DEV uint64_t f2_bits(float2 a) { return (uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32); }
CN_DEV float2 f2_of(uint64_t r) { return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32))); }
CN_DEV float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return f2_of(r);
}
CN_DEV float2 add2(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_of(r);
}
CN_DEV float2 mul2(float2 a, float2 b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_of(r);
}
CN_DEV float2 f2(float v) { return make_float2(v, v); }
// gelu_erf of two values, with the same operations (and so the same bits)
// as gelu_erf on each.
CN_DEV float2 gelu_erf2(float2 v) {
    const float2 av = make_float2(fabsf(v.x), fabsf(v.y));
    const float2 d = fma2(f2(CN_AS_P * 0.70710678118654752f), av, f2(1.0f));
    const float2 t = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    float2 y = fma2(t, f2(0.5f * CN_AS_A5), f2(0.5f * CN_AS_A4));
    y = fma2(t, y, f2(0.5f * CN_AS_A3));
    y = fma2(t, y, f2(0.5f * CN_AS_A2));
    y = fma2(t, y, f2(0.5f * CN_AS_A1));
    y = mul2(y, t);
    const float2 q = mul2(v, mul2(v, f2(-0.5f * 1.4426950408889634f)));
    const float2 e = make_float2(ex2_approx(q.x), ex2_approx(q.y));
    return fma2(make_float2(-av.x, -av.y), mul2(y, e), make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f)));
}
CN_DEV float apply_act(int act, float v) {
    if (act == ACT_HARDSWISH) return hardswish(v);
    if (act == ACT_GELU) return gelu_erf(v);
    return v;
}

// ---- running statistics ------------------------------------------------------
// (count, mean, M2) triples merged with the pairwise update of Chan et al.:
//   n = na + nb, d = mb - ma, mean = ma + d nb / n, M2 = M2a + M2b + d^2 na nb / n.
// Merging in a fixed order makes every reduction deterministic.
template <typename T>
struct Moments {
    T n, mean, m2;
};
template <typename T>
CN_DEV Moments<T> merge(Moments<T> a, Moments<T> b) {
    T n = a.n + b.n;
    if (n == T(0)) return a;
    T d = b.mean - a.mean;
    T fb = b.n / n;
    Moments<T> r;
    r.n = n;
    r.mean = a.mean + d * fb;
    r.m2 = a.m2 + b.m2 + d * d * a.n * fb;
    return r;
}
// Shifted power sums (count, S1 = sum(v - K), S2 = sum((v - K)^2)) with a
// shift K close to the data: summed with plain additions (a butterfly of
// commutative adds gives every lane the identical result), converted to
// (count, mean, M2) once, in fp64, as mean = K + S1/n, M2 = S2 - S1^2/n.
CN_DEV float3 warp_sum3(float3 v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, off);
    }
    return v;
}
// (count, mean, M2) of one channel from its per_c partials (count, K, S1,
// S2), each a sum about its own shift K, one of its own values: the partials
// move to one common shift K0 (the first non-empty partial's, a value of the
// channel's data) by the exact identities S1' = S1 + n d, S2' = S2 + d (2 S1
// + n d), d = K - K0, which stay well conditioned since every K lies within
// a few standard deviations of the data; lanes add them in a fixed order, a
// butterfly of commutative adds gives every lane the same bits, and one
// division gives mean = K0 + S1'/n, M2 = S2' - S1'^2/n.  Deterministic.
CN_DEV Moments<float> channel_moments(const float4 *p, int per_c, int lane) {
    // common shift: the first non-empty partial's (lowest lane of the first 32)
    const float4 f = lane < per_c ? p[lane] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const unsigned has = __ballot_sync(0xffffffffu, f.x > 0.0f);
    if (!has) {
        // no non-empty partial among the first 32: take the first anywhere
        // (serially; only for channels that are empty at the start)
        float K0 = 0.0f;
        for (int i = 0; i < per_c; ++i)
            if (p[i].x > 0.0f) {
                K0 = p[i].y;
                break;
            }
        float3 v = make_float3(0.0f, 0.0f, 0.0f);
        for (int i = lane; i < per_c; i += 32) {
            const float4 q = p[i];
            const float d = q.y - K0;
            v.x += q.x;
            v.y += fmaf(q.x, d, q.z);
            v.z += fmaf(d, fmaf(q.x, d, 2.0f * q.z), q.w);
        }
        v = warp_sum3(v);
        if (!(v.x > 0.0f)) return Moments<float>{0.0f, 0.0f, 0.0f};
        const float mu_s = v.y / v.x;
        return Moments<float>{v.x, K0 + mu_s, fmaxf(v.z - v.y * mu_s, 0.0f)};
    }
    const float K0 = __shfl_sync(0xffffffffu, f.y, __ffs(has) - 1);
    float3 v = make_float3(0.0f, 0.0f, 0.0f);  // (count, S1', S2') about K0
    for (int i = lane; i < per_c; i += 32) {
        const float4 q = i == lane ? f : p[i];
        const float d = q.y - K0;
        v.x += q.x;
        v.y += fmaf(q.x, d, q.z);
        v.z += fmaf(d, fmaf(q.x, d, 2.0f * q.z), q.w);
    }
    v = warp_sum3(v);
    const float mu_s = v.y / v.x;  // mean - K0
    return Moments<float>{v.x, K0 + mu_s, fmaxf(v.z - v.y * mu_s, 0.0f)};
}

CN_DEV Moments<double> moments_from_sums(double n, double K, double s1, double s2) {
    if (n <= 0.0) return Moments<double>{0.0, 0.0, 0.0};
    const double m2 = s2 - s1 * s1 / n;
    return Moments<double>{n, K + s1 / n, m2 > 0.0 ? m2 : 0.0};
}
// Butterfly merge over the 32 lanes of a warp; every lane ends with the result.
CN_DEV Moments<float> warp_merge(Moments<float> m) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Moments<float> o;
        o.n = __shfl_xor_sync(0xffffffffu, m.n, off);
        o.mean = __shfl_xor_sync(0xffffffffu, m.mean, off);
        o.m2 = __shfl_xor_sync(0xffffffffu, m.m2, off);
        // Lower lane is always the left operand so both lanes compute the
        // same value bit for bit.
        m = ((threadIdx.x & off) == 0) ? merge(m, o) : merge(o, m);
    }
    return m;
}

// ---- cp.async (LDGSTS) staging with zero fill --------------------------------
CN_DEV uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Copies 16 bytes global -> shared; when !pred the destination is zero-filled
// and the source is not read.
CN_DEV void cp_async16(void *smem, const void *gmem, bool pred) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(pred ? 16 : 0));
}
CN_DEV void cp_async4(void *smem, const void *gmem, bool pred) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(pred ? 4 : 0));
}
CN_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
CN_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }
CN_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::); }

CN_DEV double ldcg_f64(const double *p) { return __ldcg(p); }

// ---- mbarrier + TMA (bulk async copies) -----------------------------------------
// Error codes a kernel writes to the plan's flag.
enum { ERR_NONE = 0, ERR_TIMEOUT = 1, ERR_CHECK = 2 };

CN_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// Makes barrier initialisation visible to the async (TMA) proxy.
CN_DEV void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared accesses before its
// later async-proxy (TMA) accesses.
CN_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
CN_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
CN_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
CN_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// try_wait that lets the hardware suspend the thread until the phase
// completes or about hint_ns pass, instead of returning at once: a waiting
// warp then takes no issue slots from the warps that work.
CN_DEV bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the phase with the given parity (try_wait may
// suspend the thread for a while; a loop polling two barriers must not).
CN_DEV bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
CN_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
// Waits for the barrier phase with the given parity, giving up after
// limit_ns nanoseconds of GPU wall time.  Returns false on timeout.
CN_DEV bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) return false;
    }
}
// Records an error code (first writer wins).
CN_DEV void flag_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}
// Bounds checks of the checked build (-DCN_CHECKS, a stand-in for a memory
// checker): CN_CHECK(cond, err) is cond, and when cond fails it records
// ERR_CHECK (CN_ERR_DEVICE_CHECK) in the flag, so the caller skips the
// access.  Normal builds compile every check to true.
#ifdef CN_CHECKS
#define CN_CHECK(cond, err) ((cond) ? true : (::cn::flag_error((err), ::cn::ERR_CHECK), false))
#else
#define CN_CHECK(cond, err) true
#endif
// Tiled 4-D tensor copy global -> shared, completion counted on bar.
CN_DEV void tma_load_4d(void *smem_dst, const void *tmap, int c0, int c1, int c2, int c3,
                        uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}
// Tiled 5-D tensor copy global -> shared, completion counted on bar.
CN_DEV void tma_load_5d(void *smem_dst, const void *tmap, int c0, int c1, int c2, int c3, int c4,
                        uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(smem_u32(bar))
        : "memory");
}
// Contiguous bulk copy global -> shared (16-byte aligned addresses, size a
// multiple of 16), completion counted on bar.
CN_DEV void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace cn
