// Device helpers of the verify kernels: counter-based random numbers, the
// streaming loads, NaN-propagating max, base-2 exponentials and the merge of
// partial softmax statistics.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// --------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): each round multiplies words 0 and 2 by the two
// Philox constants, swaps the high/low halves into a new 4-word counter and
// mixes in the key; the key advances by the golden-ratio Weyl increments
// between rounds.
// --------------------------------------------------------------------------
struct Words4 {
    uint32_t w0, w1, w2, w3;
};

__device__ __forceinline__ Words4 philox10(Words4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a = 0xD2511F53u, b = 0xCD9E8D57u;
        uint32_t hi_a = __umulhi(a, c.w0), lo_a = a * c.w0;
        uint32_t hi_b = __umulhi(b, c.w2), lo_b = b * c.w2;
        c = Words4{hi_b ^ c.w1 ^ k0, lo_b, hi_a ^ c.w3 ^ k1, lo_a};
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Uniforms of draft position `pos` of sequence id `seq`: u (accept test) from
// word 0 and u2 (residual or bonus draw) from word 1, on the 2^-24 grid.
__device__ __forceinline__ void position_uniforms(uint64_t seed, uint64_t seq, uint32_t pos,
                                                  float& u, float& u2) {
    Words4 w = philox10(Words4{pos, (uint32_t)seq, (uint32_t)(seq >> 32), 0u}, (uint32_t)seed,
                        (uint32_t)(seed >> 32));
    u = (float)(w.w0 >> 8) * 5.9604644775390625e-08f;   // 2^-24
    u2 = (float)(w.w1 >> 8) * 5.9604644775390625e-08f;
}

// --------------------------------------------------------------------------
// Arithmetic helpers.
// --------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that returns NaN when either input is NaN (fmaxf drops NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ bool is_nan(float x) { return x != x; }

// Every CTA of a cluster must have started before any of them accesses
// another's shared memory. A kernel announces its start as its first
// instruction (every thread, no ordering) and waits for the whole cluster's
// announcements just before its first remote access; both run exactly once
// per thread, so the barrier phase always completes, and by then it has.
__device__ __forceinline__ void cluster_arrive_started() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_started() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their memory is visible (returns at once when the
// launch had no such dependency); let the next grid on the stream launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// --------------------------------------------------------------------------
// Streaming loads: read-only path, no L1 allocation (each byte is used once).
// --------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// --------------------------------------------------------------------------
// Partial softmax statistics in the base-2 domain. With c = log2(e) / T, a
// partial over a set of logits l is (R, s): R an integer-valued float with
// max(l * c) - 13 < R <= ceil(max(l * c)), s = sum 2^(l * c - R) (R tracks
// the maximum only as closely as keeps every term below 2^13). Because every
// R is an integer, two partials merge by an exact power-of-two rescale.
// Invalid partials carry R = NaN or R = +inf; an empty one is (-inf, 0).
// --------------------------------------------------------------------------
struct SoftPart {
    float R, s;
};

// 2^d for the integer differences d <= 0 of two partials' R (or -inf): the
// ex2 instruction returns exact powers of two for integer arguments (checked
// on sm_103a for every integer in [-160, 95]; below 2^-126 it flushes to 0).
// Every step is a select, not a branch: a merge sits on the critical path of
// the warp, CTA and cluster reductions.
__device__ __forceinline__ SoftPart merge_soft(SoftPart a, SoftPart b) {
    const float R = fmaxf(a.R, b.R);
    const float sa = a.R == -INFINITY ? 0.0f : a.s * ex2(a.R - R);
    const float sb = b.R == -INFINITY ? 0.0f : b.s * ex2(b.R - R);  // +inf: inf - inf = NaN
    const bool nan = is_nan(a.R) || is_nan(b.R);
    return SoftPart{nan ? __int_as_float(0x7fc00000) : R, nan ? 0.0f : sa + sb};
}

// Greedy partial: the largest logit and its lowest index (NaN is sticky).
struct ArgPart {
    float v;
    int i;
};

__device__ __forceinline__ ArgPart merge_arg(ArgPart a, ArgPart b) {
    const bool an = is_nan(a.v), bn = is_nan(b.v);
    const bool take_b = bn ? (!an || b.i < a.i) : (!an && (b.v > a.v || (b.v == a.v && b.i < a.i)));
    return take_b ? b : a;
}

// --------------------------------------------------------------------------
// Float-float sums (hi + lo, about 48 significant bits) for the draw's
// cumulative masses: the same role double would play, at fp32 latency (fp64
// is a slow, long-latency path on this part).
// --------------------------------------------------------------------------
struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff ff_from(float x) { return ff{x, 0.0f}; }

// s + e = a + b exactly (Knuth's two-sum).
__device__ __forceinline__ ff two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return ff{s, e};
}

// Renormalise hi + lo with |hi| >= |lo| (Dekker's fast two-sum).
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return ff{s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
    const ff s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ ff ff_add(ff a, float b) { return ff_add(a, ff{b, 0.0f}); }

__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }

// a * u for a float u.
__device__ __forceinline__ ff ff_mul(ff a, float u) {
    const float p = __fmul_rn(a.hi, u);
    const float e = __fmaf_rn(a.hi, u, -p);
    return fast_two_sum(p, __fmaf_rn(a.lo, u, e));
}

// a > b, decided on the float-float difference.
__device__ __forceinline__ bool ff_gt(ff a, ff b) {
    const ff d = ff_add(a, ff_neg(b));
    return d.hi > 0.0f || (d.hi == 0.0f && d.lo > 0.0f);
}

__device__ __forceinline__ ff ff_shfl_xor(ff a, int o) {
    return ff{__shfl_xor_sync(0xFFFFFFFFu, a.hi, o), __shfl_xor_sync(0xFFFFFFFFu, a.lo, o)};
}
__device__ __forceinline__ ff ff_shfl_up(ff a, int o) {
    return ff{__shfl_up_sync(0xFFFFFFFFu, a.hi, o), __shfl_up_sync(0xFFFFFFFFu, a.lo, o)};
}
__device__ __forceinline__ ff ff_shfl(ff a, int l) {
    return ff{__shfl_sync(0xFFFFFFFFu, a.hi, l), __shfl_sync(0xFFFFFFFFu, a.lo, l)};
}

// Rows of one sequence share one 8-byte slot per row in shared memory; the
// two views are stored through the same float2.
__device__ __forceinline__ float2 pack(SoftPart p) { return make_float2(p.R, p.s); }
__device__ __forceinline__ float2 pack(ArgPart p) { return make_float2(p.v, __int_as_float(p.i)); }
__device__ __forceinline__ SoftPart as_soft(float2 f) { return SoftPart{f.x, f.y}; }
__device__ __forceinline__ ArgPart as_arg(float2 f) { return ArgPart{f.x, __float_as_int(f.y)}; }

}  // namespace sv

namespace sv {

// --------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA, non-tensor, no multicast) wrappers.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete, giving up
// after `limit` polls (each poll may suspend the thread for a short,
// hardware-chosen time). Returns false on giving up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Bulk copy of `bytes` (a multiple of 16) from global to this CTA's shared
// memory; both addresses 16-byte aligned. Completion is signalled on `bar`
// as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// An L2 policy under which the lines a copy brings in are evicted before any
// others. The logits each pass through L2 once per call; a call streams more
// bytes than L2 holds, and under the default policy that stream also evicts
// the kernel's own instructions, whose once-per-call phases (decision, final
// draw) then fetch them from HBM.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy (l2_evict_first_policy).
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gsrc, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

}  // namespace sv

namespace sv {

// --------------------------------------------------------------------------
// Packed fp32x2 arithmetic (two IEEE round-to-nearest operations per
// instruction, sm_100 and later). A pair lives in one 64-bit register.
// --------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float a, float b) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack2(f32x2 r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 2^x of both halves (two MUFU operations).
__device__ __forceinline__ f32x2 ex2x2(f32x2 x) {
    float a, b;
    unpack2(x, a, b);
    return pack2(ex2(a), ex2(b));
}

// Element pair of a 32-bit word: bf16 x2 widened exactly, low half first.
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) {
    return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

}  // namespace sv

namespace sv {

// Orders this thread's earlier generic-proxy shared-memory accesses before
// its later async-proxy ones (a bulk copy that overwrites what was just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace sv
