// bn_device.cuh -- the main kernel template of libbeamnorm (sm_103a) and the
// arithmetic helpers it shares with the small-T finalize (bn_wide.cu).
//
// Operation: the arithmetic epilogue of a fused tensor-parallel all-reduce
// ("Fuse Beam's TP all-reduce with its sandwich norms", vLLM pull request
// 62366, section Claims: FP32 norm-residual-norm epilogue, optional MoE
// finalize before the reduction keeping the local BF16 rounding; section
// Details: no FMA contraction of the FP32 epilogue, so this file is compiled
// with -fmad=false), and its variants from sglang pull request 34134 (description:
// the plain all-reduce / residual / RMSNorm pattern and the MoE pattern with
// the finalize and shared-expert add folded in ahead of it).
//
// Design (GB300):
//   * One token row is owned by one CTA, or by a thread-block cluster of up to
//     16 CTAs that split the row into contiguous 16-byte-chunk slices (small T,
//     so that many SMs pull one row).  Clusters are persistent and grid-stride
//     over rows.
//   * A producer warp streams every row the CTA needs (R shard rows, or R*k
//     gathered expert rows plus R shared rows, then the residual row) from HBM
//     into a ring of shared-memory stages with 1-D TMA bulk copies
//     (cp.async.bulk, completion counted on an mbarrier).  The ring keeps
//     ~100-200 KB in flight per SM and runs ahead across row boundaries, so the
//     two row-wide reductions of one row overlap the loads of the next.
//   * Consumer warps own 16-byte chunks of the slice, read them from shared
//     memory, and do all arithmetic in registers: exact BF16 widening, the
//     rank-ordered FP32 sum, the per-shard finalize, both RMSNorms, and 16-byte
//     coalesced stores of the BF16 outputs.
//   * A sum of squares is accumulated as a compensated pair (exact products via
//     one explicit fma for the error term, two-sum for the additions), combined
//     in a fixed warp/block/cluster tree, and rounded once: as accurate as a
//     sum in twice the precision (typically within sqrt(n) * 2^-48 relative
//     of the exact sum before the final rounding), so it is the FP32 rounding
//     of the exact sum except right at a rounding boundary; a sum beyond the
//     FP32 range is +inf.
//   * Cluster partial sums (and the shard split's z rows) travel through
//     distributed shared memory as st.async remote stores whose completion
//     the receiving CTA's mbarrier counts in bytes -- no global scratch.
//   * Every wait is bounded (SM cycles and polls); on expiry the kernel records an
//     error bit, stops issuing copies, drains the copies it has in flight, runs
//     the rest of its control flow without waiting on the copy pipeline and
//     without storing (the cluster exchanges, which every CTA still feeds, are
//     still waited for), and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "bn_internal.h"

namespace bn {
namespace dev {

// A wait gives up after 2^29 SM cycles (about 0.26 s at 2 GHz) or 2^26 polls.
constexpr long long kWaitLimitCycles = 1ll << 29;
constexpr uint32_t kMaxSpins = 1u << 26;
constexpr unsigned kErrPerm = 1u;
constexpr unsigned kErrTimeout = 2u;

// ---- PTX wrappers -------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ncluster_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Acquire at cluster scope: pairs with the remote release-arrive of the
// partial-sum exchange.
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Non-suspending probes of the same phases (used when spin_wait is set).
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_probe_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Asynchronous remote store of 16 bytes into another CTA's shared memory; its
// completion counts 16 bytes on that CTA's mbarrier (addresses from mapa).
__device__ __forceinline__ void st_async_u4(uint32_t addr, const uint4 &v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
                 : "memory");
}
// Asynchronous remote store of a float pair into another CTA's shared memory;
// its completion counts 8 bytes on that CTA's mbarrier (addresses from mapa).
__device__ __forceinline__ void st_async_f2(uint32_t addr, float x, float y, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                     addr),
                 "f"(x), "f"(y), "r"(bar)
                 : "memory");
}
// 1-D TMA bulk copy global -> this CTA's shared memory, completion counted in
// bytes on the mbarrier.  dst, src and bytes are multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Programmatic dependent launch (sm_90 and later).  wait: block until every
// grid this one depends on has completed and its memory is visible (a no-op
// when the launch did not ask for programmatic serialization).  launch_dependents:
// allow the next grid in the stream to be scheduled early; it still runs no
// memory operation before its own wait.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Named barrier among the consumer warps only (the producer warp runs free).
__device__ __forceinline__ void consumer_sync(int nthreads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// ---- bounded waits --------------------------------------------------------------

// Abort bits of a CTA (a shared-memory word).
constexpr int kAbortPipe = 1;   // a wait expired: stop issuing copies, stop storing
constexpr int kAbortDsmem = 2;  // a cluster exchange itself expired: stop waiting on exchanges

struct Ctl {
    volatile int *abort;  // shared abort bits of this CTA
    unsigned *err;        // device error word
    bool spin;            // poll with test_wait instead of the suspending try_wait
    uint32_t pipe_polls;  // polls after which a pipeline wait gives up
};

// Kinds of wait.
//   kPipe:  the copy pipeline (stage and metadata barriers).  Returns false at
//           once while the CTA is aborting; gives up after ctl.pipe_polls polls
//           (normally 2^26) or 2^29 SM cycles.
//   kDsmem: the cluster exchanges (sums of squares, shard-split z rows).  They
//           are waited for even while the CTA aborts -- every CTA still sends
//           what it owes, so they complete, and no remote store may still be in
//           flight into a CTA that stops waiting -- unless an exchange itself
//           expired.
//   kDrain: the producer's final wait for its copies in flight; never skipped.
enum WaitKind { kPipe = 0, kDsmem = 1, kDrain = 2 };

template <bool CLUSTER_ACQUIRE>
__device__ __forceinline__ bool phase_done(uint32_t bar, uint32_t parity, bool spin)
{
    if (spin) return CLUSTER_ACQUIRE ? mbar_probe_cluster(bar, parity) : mbar_probe(bar, parity);
    return CLUSTER_ACQUIRE ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity);
}

// Wait for the phase of `bar` with parity `parity` to complete.  Returns false
// without waiting when the CTA's abort bits say this kind of wait is skipped,
// or after the kind's limit, in which case it records the timeout and sets the
// abort bits.  The clock is read only after 1024 unsuccessful polls: a wait
// that ends quickly costs nothing but the polls themselves.
template <bool CLUSTER_ACQUIRE, int KIND>
__device__ __forceinline__ bool wait_phase_loop(uint32_t bar, uint32_t parity, volatile int *abort,
                                                unsigned *err, bool spin, uint32_t pipe_polls)
{
    constexpr int kSkipOn = KIND == kPipe ? kAbortPipe : KIND == kDsmem ? kAbortDsmem : 0;
    if (kSkipOn != 0 && (*abort & kSkipOn)) return false;
    const uint32_t limit = KIND == kPipe ? pipe_polls : kMaxSpins;
    long long t0 = 0;
    for (uint32_t i = 1; i < limit; ++i) {
        if (phase_done<CLUSTER_ACQUIRE>(bar, parity, spin)) return true;
        if ((i & 1023u) == 0u) {
            if (kSkipOn != 0 && (*abort & kSkipOn)) return false;
            if (i == 1024u)
                t0 = clock64();
            else if (clock64() - t0 > kWaitLimitCycles)
                break;
        }
    }
    atomicOr(err, kErrTimeout);
    atomicOr(const_cast<int *>(abort), KIND == kDsmem ? (kAbortPipe | kAbortDsmem) : kAbortPipe);
    return false;
}

// The polling loop as a function of its own.  Inlined at every wait it added
// about 9 KB (11 %) to the finalize kernels' code, which is already larger
// than the SM's fastest instruction cache (a loop body of 31 KB ran at full
// rate on GB300, one of 61 KB at half); out of line, the finalize calls at
// few rows ran 3 to 4.5 % faster.  A call costs nothing while the phase is
// already complete, but the call's register convention made the 4-chunk
// reduce kernels spill, so they keep it inline (OUTLINE below).
template <bool CLUSTER_ACQUIRE, int KIND>
__device__ __noinline__ bool wait_phase_poll(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned *err, bool spin, uint32_t pipe_polls)
{
    return wait_phase_loop<CLUSTER_ACQUIRE, KIND>(bar, parity, abort, err, spin, pipe_polls);
}

template <bool CLUSTER_ACQUIRE, int KIND, bool OUTLINE = true>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl &c)
{
    // a completed phase returns at once (its data is valid even in a CTA that
    // is aborting); the abort bits are read only when the wait must poll
    if (phase_done<CLUSTER_ACQUIRE>(bar, parity, c.spin)) return true;
    if constexpr (OUTLINE)
        return wait_phase_poll<CLUSTER_ACQUIRE, KIND>(bar, parity, c.abort, c.err, c.spin, c.pipe_polls);
    else
        return wait_phase_loop<CLUSTER_ACQUIRE, KIND>(bar, parity, c.abort, c.err, c.spin, c.pipe_polls);
}

// ---- arithmetic helpers ----------------------------------------------------------
//
// The consumers work on packed FP32 pairs (f2): Blackwell's add/sub/mul .f32x2
// round each lane to nearest even exactly like the scalar instructions, so the
// results are those of the scalar definition while fewer instructions issue.
// Element 2i of a 16-byte chunk is the low lane of pair i.
//
// One rule keeps the arithmetic uncontracted: ptxas fuses a packed multiply
// that feeds a packed add into a packed fused multiply-add even under
// --fmad=false (measured: every differing result matched the fused one),
// while a scalar mul.rn.f32 feeding a packed add is left alone.  So every
// product that is later added (finalize weights, squares, the post-norm
// output before the residual add) is formed lane by lane with mul_sep2;
// packed multiplies (mul2) only feed other multiplies or outputs.

typedef unsigned long long f2;

__device__ __forceinline__ f2 f2_make(float lo, float hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b)
{
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// A product that will be added to something: two scalar multiplies, which the
// code generator keeps separate from the following addition.
__device__ __forceinline__ float mul_sep(float a, float b)
{
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ f2 mul_sep2(f2 a, f2 b)
{
    float a0, a1, b0, b1;
    f2_split(a, a0, a1);
    f2_split(b, b0, b1);
    return f2_make(mul_sep(a0, b0), mul_sep(a1, b1));
}
// Only used to obtain the exact rounding error of a product (see acc_square2).
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// -(a * b) rounded once (round to nearest even is symmetric, so this is the
// negated product exactly); the negation is an operand modifier of the scalar
// multiply, not an instruction of its own.
__device__ __forceinline__ float mul_neg(float a, float b)
{
    float r;
    asm("{\n\t.reg .f32 t;\n\tneg.f32 t, %2;\n\tmul.rn.f32 %0, %1, t;\n\t}" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Exact widening of a word holding two BF16 values (low half -> low lane).
__device__ __forceinline__ f2 widen2(uint32_t w)
{
    return f2_make(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ void widen8(const uint4 &v, f2 *x)
{
    x[0] = widen2(v.x);
    x[1] = widen2(v.y);
    x[2] = widen2(v.z);
    x[3] = widen2(v.w);
}

// s[m] += the BF16 pair in word m of v, lane by lane, with PTX's mixed-precision
// add (sm_100 and later): it converts the BF16 operand exactly and rounds the
// sum once, the result of widening and then adding, in one instruction per
// element instead of one and a half.
__device__ __forceinline__ float add_bf16_lo(float c, uint32_t w)
{
    float r;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, lo, %1; }"
        : "=f"(r)
        : "f"(c), "r"(w));
    return r;
}
__device__ __forceinline__ float add_bf16_hi(float c, uint32_t w)
{
    float r;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, hi, %1; }"
        : "=f"(r)
        : "f"(c), "r"(w));
    return r;
}
__device__ __forceinline__ void add_bf16x8(f2 *s, const uint4 &v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float lo, hi;
        f2_split(s[m], lo, hi);
        s[m] = f2_make(add_bf16_lo(lo, w[m]), add_bf16_hi(hi, w[m]));
    }
}

// Round a pair to BF16 (nearest even) and pack it, low lane in the low half.
__device__ __forceinline__ uint32_t round2(f2 v)
{
    float lo, hi;
    f2_split(v, lo, hi);
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ uint4 round8(const f2 *v)
{
    return make_uint4(round2(v[0]), round2(v[1]), round2(v[2]), round2(v[3]));
}

// s + e == a + b exactly (Knuth's two-sum; no ordering assumption).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Two independent compensated accumulators (one per lane): (S, E) += x*x.
// The product's rounding error comes from one explicit fma (it only measures
// the error of the rounded product; no result value is contracted) and the
// addition's error from two-sum; both are carried in E.  The product is
// formed negated, np = -p, which the fma needs as its addend: the two-sum is
// then written with np, S - np = S + p and -(np + bb) = p - bb, the same
// roundings of the same values.
__device__ __forceinline__ void acc_square2(f2 &S, f2 &E, f2 x)
{
    float x0, x1;
    f2_split(x, x0, x1);
    const f2 np = f2_make(mul_neg(x0, x0), mul_neg(x1, x1));
    const f2 pe = fma2(x, x, np);
    const f2 s = sub2(S, np);
    const f2 bb = sub2(s, S);
    const f2 e = sub2(sub2(S, sub2(s, bb)), add2(np, bb));
    S = s;
    E = add2(E, add2(e, pe));
}

// One compensated accumulator: (S, E) += x*x, as acc_square2 lane by lane.
__device__ __forceinline__ void acc_square1(float &S, float &E, float x)
{
    const float p = mul_sep(x, x);
    const float pe = fmaf(x, x, -p);
    float s, e;
    two_sum(S, p, s, e);
    S = s;
    E = E + (e + pe);
}

// (S, E) += (lo * up)^2 + (hi * up)^2 for the two values of v, scaled by a
// power of two (exact); the second pass of a row of tiny values, kept scalar
// so that the rare path holds few registers.
__device__ __forceinline__ void acc_square_scaled(float &S, float &E, f2 v, float up)
{
    float lo, hi;
    f2_split(v, lo, hi);
    acc_square1(S, E, mul_sep(lo, up));
    acc_square1(S, E, mul_sep(hi, up));
}

// (S, E) += (S2, E2) for two compensated sums of squares.  Both running parts
// are non-negative, so the larger one is known without a branch and Dekker's
// fast two-sum (the smaller part minus what the rounded sum kept of it) gives
// the exact rounding error, the value two-sum gives, in a chain of three
// dependent operations instead of five.  The sum itself is formed from S and
// S2, so a NaN in either still reaches it.
__device__ __forceinline__ void combine(float &S, float &E, float S2, float E2)
{
    const float s = S + S2;
    const float hi = fmaxf(S, S2);
    const float lo = fminf(S, S2);
    const float e = lo - (s - hi);
    S = s;
    E = (E + E2) + e;
}

// Fold the two lanes of a packed accumulator into one (S, E), low lane first.
__device__ __forceinline__ void fold2(f2 S2, f2 E2, float &S, float &E)
{
    float s0, s1, e0, e1;
    f2_split(S2, s0, s1);
    f2_split(E2, e0, e1);
    S = s0;
    E = e0;
    combine(S, E, s1, e1);
}

// The rounded value of a compensated pair.  A sum of non-negative squares
// whose running part S has left the FP32 range is +inf (NaN if an operand was
// NaN); its error part E then holds inf - inf = NaN, so S itself is the
// result -- as for the exactly accumulated sum rounded once.
__device__ __forceinline__ float pair_value(float S, float E)
{
    return S < __int_as_float(0x7f800000) ? S + E : S;
}

// A compensated sum of squares is exact only while the squares stay in FP32's
// normal range: below it a square's rounding error cannot be represented.  A
// row whose sum is below 2^-80 (every value below 2^-40) is therefore summed
// again with each value scaled by 2^k, exactly (a power of two); the scaled
// sum lands in [0.5, 2), and the result is scaled back by 2^-k twice.  A sum
// that is zero or subnormal (every value below 2^-63) takes k = 100, which
// lifts every nonzero FP32 value's square above 2^-100.  In the scaled pass
// only a value over 2^51 times smaller than the row's largest can lose its
// square's error term, an error below 2^-148 of the scaled sum.
__device__ __forceinline__ bool needs_rescale(float ss) { return ss < __int_as_float(0x17800000); }

__device__ __forceinline__ int rescale_exp(float ss)
{
    const int e = (int)((__float_as_uint(ss) >> 23) & 0xffu);  // biased exponent, ss >= 0
    return e == 0 ? 100 : (127 - e) >> 1;
}

__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }

__device__ __forceinline__ void warp_tree(float &S, float &E)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float S2 = __shfl_down_sync(0xffffffffu, S, off);
        const float E2 = __shfl_down_sync(0xffffffffu, E, off);
        combine(S, E, S2, E2);
    }
}

// The pairs src[0..n-1] (1 <= n <= 32) combined as warp_tree combines them on
// lane 0 with the lanes from n on holding zero pairs, then broadcast to every
// lane.  A zero pair changes nothing under combine, and at a level whose
// offset is n or more lane 0's partner holds only zeros, so those levels are
// left out (a CTA of 5 consumer warps runs 3 of the 5).
__device__ __forceinline__ void small_tree(const float2 *src, int n, int lane, float &S, float &E)
{
    const float2 v = lane < n ? src[lane] : make_float2(0.f, 0.f);
    S = v.x;
    E = v.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (off < n) {
            const float S2 = __shfl_down_sync(0xffffffffu, S, off);
            const float E2 = __shfl_down_sync(0xffffffffu, E, off);
            combine(S, E, S2, E2);
        }
    }
    S = __shfl_sync(0xffffffffu, S, 0);
    E = __shfl_sync(0xffffffffu, E, 0);
}

// 1 / sqrt(ss / H + eps): three correctly rounded FP32 operations
// (-prec-div and -prec-sqrt are left at their IEEE defaults).
__device__ __forceinline__ float rms_factor(float ss, int H, float eps)
{
    const float mean = ss / (float)H;
    return 1.0f / sqrtf(mean + eps);
}

// ---- the kernel ------------------------------------------------------------------

struct Smem {
    uint8_t *stages;
    uint32_t stages_u32;
    uint32_t full0, empty0, mfull0, mempty0, ex0;  // mbarrier addresses (8 bytes apart)
    float2 *red;                                   // [2][32]
    float2 *xslot;                                 // [2][kMaxCluster]
    int32_t *mperm;                                // [2][kMaxMeta]
    float *mw;                                     // [2][kMaxMeta]
};

// Row-wide sum of squares: compensated pairs reduced over the warp, the
// consumer warps of the CTA, then the CTAs of the cluster, in a fixed order;
// every consumer thread of every CTA of the cluster gets the same value.
// TREE: the CTAs' pairs are combined by a tree, not one after the other
// (taken by the shard-split kernels: C4 at T=16 13.24 -> 12.88 us, C3 at
// T=16 11.23 -> 10.79; the column-split kernels were 0.5-1 % slower with it,
// their code being laid out differently at the register cap).
template <bool OUTLINE, bool TREE>
__device__ __forceinline__ float row_sum_squares(f2 S2, f2 E2, int &nred, const Smem &sm,
                                                 uint32_t cs, uint32_t q, int NT, int NW,
                                                 int warp, int lane, int tid, const Ctl &ctl,
                                                 bool &live)
{
    float S, E;
    fold2(S2, E2, S, E);
    warp_tree(S, E);
    const int b = nred & 1;
    if (lane == 0) sm.red[b * 32 + warp] = make_float2(S, E);
    consumer_sync(NT);
    small_tree(sm.red + b * 32, NW, lane, S, E);
    if (cs > 1) {
        float2 *slots = sm.xslot + b * kMaxCluster;
        const uint32_t bar = sm.ex0 + 8u * (uint32_t)b;
        // Thread d stores this CTA's pair into slot q of CTA d with one
        // asynchronous remote store that counts 8 bytes on CTA d's barrier;
        // each CTA's own arrive expects cs * 8 bytes.  The cs sends overlap and
        // need no fence (one thread storing and release-arriving for every
        // CTA in turn cost ~2.3 us per exchange at cs = 8 on GB300).
        if (tid == 0) mbar_arrive_expect_tx(bar, 8u * cs);
        if (tid < (int)cs) {
            const uint32_t d = (uint32_t)tid;
            st_async_f2(mapa(smem_addr(slots + q), d), S, E, mapa(bar, d));
        }
        if (!wait_phase<true, kDsmem, OUTLINE>(bar, (uint32_t)(nred >> 1) & 1u, ctl)) live = false;
        if constexpr (TREE) {
            small_tree(slots, (int)cs, lane, S, E);
        } else {
            S = slots[0].x;
            E = slots[0].y;
            for (uint32_t c = 1; c < cs; ++c) combine(S, E, slots[c].x, slots[c].y);
        }
    }
    ++nred;
    return pair_value(S, E);
}

// SPLITR (finalize modes only): the cs CTAs of a cluster split a token row by
// shard instead of by columns (cs divides R).  CTA q finalizes shards
// q * R/cs .. (q + 1) * R/cs - 1 over the whole row ((k + 1) * R/cs copies
// instead of R * (k + 1)) and sends every chunk of each BF16 result z_r to
// the CTA whose column slice holds it; each CTA then sums the R z rows of its
// slice in rank order and runs the epilogue on the slice exactly as in the
// column split.
// FULL: every consumer thread owns exactly CPT chunks of every slice it
// works on (the host launches it only when slice == CPT * consumers for all
// CTAs), so the per-chunk bounds checks drop out of the loops.  In the shard
// split it covers the finalize over the whole row (nchunks == CPT *
// consumers); the epilogue slice there stays checked.
template <int MODE, int CPT, bool SPLITR, bool FULL, bool TINY>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) bn_kernel(const Args a)
{
    constexpr bool FIN = (MODE & F_FIN) != 0;
    constexpr bool SUM_IN = (MODE & F_SUM_IN) != 0;
    constexpr bool POSTNORM = (MODE & F_POSTNORM) != 0;
    constexpr bool RESNORM = (MODE & F_RESNORM) != 0;
    constexpr bool SUM_OUT = (MODE & F_SUM_OUT) != 0;
    constexpr bool Z_OUT = (MODE & F_Z_OUT) != 0;
    constexpr bool REDUCE = !Z_OUT;
    // the waits' polling loops out of line, except in the 4-chunk kernels,
    // whose registers the call's convention would spill
    constexpr bool kOutline = CPT < 4;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;

    const SmemLayout L = SmemLayout::make(a.stages, a.stage_bytes, a.gamma_bytes, a.zbuf_bytes, FIN);
    Smem sm;
    sm.stages = smem + L.stages_off;
    sm.stages_u32 = smem_addr(sm.stages);
    sm.full0 = smem_addr(smem + L.bars_off);
    sm.empty0 = sm.full0 + 8u * (uint32_t)a.stages;
    sm.mfull0 = sm.empty0 + 8u * (uint32_t)a.stages;
    sm.mempty0 = sm.mfull0 + 16u;
    sm.ex0 = sm.mempty0 + 16u;
    sm.red = reinterpret_cast<float2 *>(smem + L.red_off);
    sm.xslot = reinterpret_cast<float2 *>(smem + L.xslot_off);
    sm.mperm = reinterpret_cast<int32_t *>(smem + L.meta_off);
    sm.mw = reinterpret_cast<float *>(smem + L.meta_off + 2u * kMaxMeta * 4u);

    const int NT = (int)blockDim.x - 32;  // consumer threads
    const int NW = NT >> 5;
    const int tid = (int)threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t cs = cluster_nctarank();
    const uint32_t q = cluster_ctarank();
    const int cl = (int)cluster_id_x();
    const int ncl = (int)ncluster_x();
    // The shard split needs a cluster size that divides R (the host launches
    // it so); any other shape returns at once, before any barrier.
    if (SPLITR && (a.R % (int)cs) != 0) {
        griddep_wait();
        if (threadIdx.x == 0) atomicOr(a.err, kErrTimeout);
        return;
    }
    // this CTA's slice of the row: chunks [c0, c0 + nch)
    const int c0 = (int)(((long long)q * a.nchunks) / (long long)cs);
    const int nch = (int)(((long long)(q + 1) * a.nchunks) / (long long)cs) - c0;
    const int S = a.stages;
    const size_t H = (size_t)a.H;
    const bool has_shared = FIN && a.shared != nullptr;

    // barriers: full[S], empty[S], meta_full[2], meta_empty[2], exchange[2], z ready
    const int nbars = 2 * S + 7;
    for (int i = tid; i < nbars; i += (int)blockDim.x) {
        uint32_t count;
        if (i < S) count = 1u;                      // full: the producer's expect-tx arrive
        else if (i < 2 * S) count = (uint32_t)NW;   // empty: one arrive per consumer warp
        else if (i < 2 * S + 2) count = 32u;        // meta_full: every producer lane
        else if (i < 2 * S + 4) count = (uint32_t)NW;  // meta_empty
        else count = 1u;                            // exchange, z ready: the owner's expect-tx arrive
        mbar_init(sm.full0 + 8u * (uint32_t)i, count);
    }
    if (tid == 0) s_abort = 0;
    fence_mbarrier_init();
    __syncthreads();
    if (cs > 1) cluster_sync_all();
    // Only shared memory was touched so far: under a programmatic launch the
    // setup above overlaps the previous kernel's tail.  No global load or store
    // comes before this wait.
    griddep_wait();
    const Ctl ctl{&s_abort, a.err, a.spin_wait != 0,
                  a.wait_polls > 0 ? (uint32_t)a.wait_polls : kMaxSpins};

    // Copies per token row ("items"), in the order both sides walk them:
    //   FIN:    for each shard r: its k gathered rows, then its shared row;
    //   reduce: the R shard rows;  norm only: the FP32 sum row;
    //   then the residual row when the epilogue runs.
    // A stage holds up to G = a.group consecutive items of one row (one
    // barrier for all of them); a row always ends on a stage boundary.
    const int per_shard = FIN ? a.k + (has_shared ? 1 : 0) : 1;
    const int spc = SPLITR ? a.R / (int)cs : a.R;  // shards per CTA (shard split)
    const int row_items = (SUM_IN ? 1 : spc * per_shard) + (RESNORM ? 1 : 0);
    const uint32_t zready = sm.ex0 + 16u;       // shard split: the z rows of all CTAs are ready
    uint4 *zbuf = reinterpret_cast<uint4 *>(smem + L.zbuf_off);
    const int G = a.group;
    const uint32_t item_bytes = (uint32_t)a.item_bytes;
    // Items per stage, from the items left in the row: up to G.  In the shard
    // split the residual copy (a column slice) is smaller than the whole-row
    // copies before it, so it takes a stage of its own.
    constexpr bool kLoneLast = SPLITR && RESNORM;
    auto items_in_stage = [&](int left) -> int {
        if (kLoneLast) {
            if (left == 1) return 1;
            --left;
        }
        return left < G ? left : G;
    };

    if (warp == NW) {
        // ================= producer warp =================
        uint32_t stage = 0, phase = 0, issued = 0;  // issued = stages armed
        int pos = 0, n_in = 0;                      // item slot in the armed stage
        bool ok = true;
        // Gather indices and weights of a row are loaded into registers one row
        // ahead (all lanes, up to 8 slots per lane), so their latency overlaps
        // the copies of the current row.
        constexpr int kMetaPerLane = kMaxMeta / 32;
        int32_t pv[kMetaPerLane];
        float wv[kMetaPerLane];
        const int nm = FIN ? a.R * a.k : 0;
        auto prefetch_meta = [&](int t) {
#pragma unroll
            for (int u = 0; u < kMetaPerLane; ++u) {
                const int i = lane + 32 * u;
                if (i < nm && t < a.T) {
                    const int r = i / a.k;
                    const int j = i - r * a.k;
                    const size_t mi = ((size_t)r * a.T + t) * a.k + j;
                    pv[u] = __ldg(a.perm + mi);
                    wv[u] = __ldg(a.w + mi);
                }
            }
        };
        if constexpr (FIN) prefetch_meta(cl);
        for (int t = cl, it = 0; t < a.T && ok; t += ncl, ++it) {
            const int slot = it & 1;
            if constexpr (FIN) {
                // publish this row's gather indices and weights (all lanes)
                bool got = true;
                if (lane == 0)
                    got = wait_phase<false, kPipe, kOutline>(sm.mempty0 + 8u * slot,
                                                  (((uint32_t)it >> 1) & 1u) ^ 1u, ctl);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) {
                    ok = false;
                    break;
                }
                const long long lim = (long long)a.T * a.k;
#pragma unroll
                for (int u = 0; u < kMetaPerLane; ++u) {
                    const int i = lane + 32 * u;
                    if (i < nm) {
                        int p = pv[u];
                        if (p < 0 || (long long)p >= lim) {
                            atomicOr(a.err, kErrPerm);
                            p = 0;
                        }
                        sm.mperm[slot * kMaxMeta + i] = p;
                        sm.mw[slot * kMaxMeta + i] = wv[u];
                    }
                }
                mbar_arrive(sm.mfull0 + 8u * slot);
                __syncwarp();
                prefetch_meta(t + ncl);
            }
            if (lane == 0) {
                int left = row_items;
                // one copy into the next item slot; a stage is armed (its
                // expected byte count set) when its first item is issued.  All
                // items of a stage have the same size (a group of more than one
                // item never holds the FP32 sum).
                auto put = [&](const void *src, uint32_t bytes) -> bool {
                    const uint32_t fb = sm.full0 + 8u * stage;
                    if (pos == 0) {
                        n_in = items_in_stage(left);
                        if (!wait_phase<false, kPipe, kOutline>(sm.empty0 + 8u * stage, phase ^ 1u, ctl)) return false;
                        mbar_arrive_expect_tx(fb, bytes * (uint32_t)n_in);
                        ++issued;
                    }
                    bulk_g2s(sm.stages_u32 + stage * (uint32_t)a.stage_bytes + (uint32_t)pos * item_bytes,
                             src, bytes, fb);
                    --left;
                    if (++pos == n_in) {
                        pos = 0;
                        if (++stage == (uint32_t)S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    return true;
                };
                const uint32_t bytes16 = (uint32_t)nch * 16u;
                const size_t col = (size_t)c0 * 8u;
                if constexpr (SUM_IN) {
                    ok = put(a.sum_in + (size_t)t * H + col, bytes16 * 2u);
                } else if constexpr (FIN && SPLITR) {
                    // this CTA's shards over the whole row
                    const int32_t *mp = sm.mperm + slot * kMaxMeta;
                    const uint32_t row_bytes = (uint32_t)a.nchunks * 16u;
                    for (int rr = 0; rr < spc && ok; ++rr) {
                        const int r = (int)q * spc + rr;
                        const uint16_t *xr = a.src + (size_t)r * a.T * a.k * H;
                        for (int j = 0; j < a.k && ok; ++j)
                            ok = put(xr + (size_t)mp[r * a.k + j] * H, row_bytes);
                        if (ok && has_shared) ok = put(a.shared + ((size_t)r * a.T + t) * H, row_bytes);
                    }
                } else if constexpr (FIN) {
                    const int32_t *mp = sm.mperm + slot * kMaxMeta;
                    for (int r = 0; r < a.R && ok; ++r) {
                        const uint16_t *xr = a.src + (size_t)r * a.T * a.k * H;
                        for (int j = 0; j < a.k && ok; ++j)
                            ok = put(xr + (size_t)mp[r * a.k + j] * H + col, bytes16);
                        if (ok && has_shared)
                            ok = put(a.shared + ((size_t)r * a.T + t) * H + col, bytes16);
                    }
                } else {
                    for (int r = 0; r < a.R && ok; ++r)
                        ok = put(a.src + ((size_t)r * a.T + t) * H + col, bytes16);
                }
                if constexpr (RESNORM) {
                    if (ok) ok = put(a.residual + (size_t)t * H + col, bytes16);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        // drain: wait (bounded, even when aborting) for every stage still in
        // flight, including one left partly issued by an abort
        if (lane == 0) {
            const uint32_t n = issued < (uint32_t)S ? issued : (uint32_t)S;
            uint32_t st = stage, ph = phase;
            if (pos != 0) {
                // the armed stage never completes its byte count: give its
                // issued copies the bounded time to land
                wait_phase<false, kDrain, kOutline>(sm.full0 + 8u * st, ph, ctl);
            }
            const uint32_t done_n = pos != 0 ? n - 1 : n;
            for (uint32_t i = 0; i < done_n; ++i) {
                if (st == 0) {
                    st = (uint32_t)S - 1u;
                    ph ^= 1u;
                } else {
                    --st;
                }
                wait_phase<false, kDrain, kOutline>(sm.full0 + 8u * st, ph, ctl);
            }
        }
    } else {
        // ================= consumer warps =================
        uint32_t stage = 0, phase = 0;
        int nred = 0;
        bool live = true;  // false once a wait failed: keep the control flow, store nothing
        // item cursor: a stage is waited for when its first item is taken and
        // released when its last item is done.  The reduce modes carry one
        // item per stage, so there every take waits and every release frees.
        int cpos = 0, cn = 0, cleft = 0;
        const uint8_t *cbase = sm.stages;
        auto take = [&]() -> const uint8_t * {
            if (!FIN || cpos == 0) {
                cn = items_in_stage(cleft);
                if (!wait_phase<false, kPipe, kOutline>(sm.full0 + 8u * stage, phase, ctl)) live = false;
                cbase = sm.stages + (size_t)stage * (size_t)a.stage_bytes;
            }
            return cbase + (size_t)cpos * item_bytes;
        };
        // A warp whose wait failed never releases a stage again: the producer
        // must not re-arm a stage whose copies it has not seen land (lane 0
        // saw every stage it releases complete).
        auto release = [&]() {
            --cleft;
            if (!FIN || ++cpos == cn) {
                cpos = 0;
                __syncwarp();
                if (lane == 0 && live) mbar_arrive(sm.empty0 + 8u * stage);
                if (++stage == (uint32_t)S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        };
        auto chunk = [&](const uint8_t *p, int lc) -> uint4 {
            return *reinterpret_cast<const uint4 *>(p + (size_t)lc * 16);
        };
        // Gamma slots: each consumer thread copies the gammas of its own chunks
        // into shared memory once, laid out by chunk so that a warp's 16-byte
        // reads are contiguous; it alone reads them back (no barrier needed).
        //   slot (g, half, lc) = gsm[(g * 2 + half) * gstride + lc], lc < nch
        const int gstride = a.gamma_stride;
        float4 *gsm = reinterpret_cast<float4 *>(smem + L.gamma_off);
        constexpr int kGPost = 0;
        constexpr int kGPre = POSTNORM ? 1 : 0;
        if constexpr (RESNORM) {
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int lc = tid + i * NT;
                if ((FULL && !SPLITR) || lc < nch) {
                    const float4 *gq = reinterpret_cast<const float4 *>(a.gamma_pre + (size_t)(c0 + lc) * 8);
                    gsm[(kGPre * 2 + 0) * gstride + lc] = __ldg(gq);
                    gsm[(kGPre * 2 + 1) * gstride + lc] = __ldg(gq + 1);
                    if constexpr (POSTNORM) {
                        const float4 *gp = reinterpret_cast<const float4 *>(a.gamma_post + (size_t)(c0 + lc) * 8);
                        gsm[(kGPost * 2 + 0) * gstride + lc] = __ldg(gp);
                        gsm[(kGPost * 2 + 1) * gstride + lc] = __ldg(gp + 1);
                    }
                }
            }
        }
        auto gamma8 = [&](int g, int i, f2 *out) {
            const int lc = tid + i * NT;
            const float4 x = gsm[(g * 2 + 0) * gstride + lc];
            const float4 y = gsm[(g * 2 + 1) * gstride + lc];
            out[0] = f2_make(x.x, x.y);
            out[1] = f2_make(x.z, x.w);
            out[2] = f2_make(y.x, y.y);
            out[3] = f2_make(y.z, y.w);
        };

        for (int t = cl, it = 0; t < a.T; t += ncl, ++it) {
            const int slot = it & 1;
            cleft = row_items;
            f2 s[CPT][4];
#pragma unroll
            for (int i = 0; i < CPT; ++i)
#pragma unroll
                for (int m = 0; m < 4; ++m) s[i][m] = 0ull;

            // ---- the reduced sum s (or the per-shard finalize results) ----
            if constexpr (SUM_IN) {
                const uint8_t *p = take();
#pragma unroll
                for (int i = 0; i < CPT; ++i) {
                    const int lc = tid + i * NT;
                    if ((FULL && !SPLITR) || lc < nch) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(p + (size_t)lc * 32);
                        const uint4 v = *reinterpret_cast<const uint4 *>(p + (size_t)lc * 32 + 16);
                        s[i][0] = ((f2)u.y << 32) | u.x;
                        s[i][1] = ((f2)u.w << 32) | u.z;
                        s[i][2] = ((f2)v.y << 32) | v.x;
                        s[i][3] = ((f2)v.w << 32) | v.z;
                    }
                }
                release();
            } else if constexpr (FIN && SPLITR) {
                if (!wait_phase<false, kPipe, kOutline>(sm.mfull0 + 8u * slot, ((uint32_t)it >> 1) & 1u, ctl))
                    live = false;
                const float *wrow = sm.mw + slot * kMaxMeta;
                // Each 16-byte chunk of every z_r this CTA finalizes goes
                // straight to the CTA whose column slice holds it, into row r of
                // that CTA's z buffer ([R][zstride] chunks), as an asynchronous
                // remote store counted on that CTA's z-ready barrier; each CTA
                // expects R * nch chunks of 16 bytes per token row.
                const int zstride = (a.nchunks + (int)cs - 1) / (int)cs;
                const uint32_t zb = smem_addr(zbuf);
                if constexpr (REDUCE) {
                    if (tid == 0) mbar_arrive_expect_tx(zready, (uint32_t)(a.R * nch) * 16u);
                }
                // shards q * spc .. q * spc + spc - 1, each over the whole row
                // (chunks tid + i * NT < nchunks)
                for (int rr = 0; rr < spc; ++rr) {
                    const int r = (int)q * spc + rr;
                    f2 acc[CPT][4];
#pragma unroll
                    for (int i = 0; i < CPT; ++i)
#pragma unroll
                        for (int m = 0; m < 4; ++m) acc[i][m] = 0ull;
                    // slot 0: acc = w0 * x0
                    {
                        const float w0 = wrow[r * a.k];
                        const f2 w2 = f2_make(w0, w0);
                        const uint8_t *p = take();
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            f2 x[4] = {0ull, 0ull, 0ull, 0ull};
                            if (FULL || lc < a.nchunks) widen8(chunk(p, lc), x);
#pragma unroll
                            for (int m = 0; m < 4; ++m) acc[i][m] = mul_sep2(w2, x[m]);
                        }
                        release();
                    }
                    // slots 1..k-1: acc = acc + wj * xj
#pragma unroll 2
                    for (int j = 1; j < a.k; ++j) {
                        const float wj = wrow[r * a.k + j];
                        const f2 w2 = f2_make(wj, wj);
                        const uint8_t *p = take();
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            if (FULL || lc < a.nchunks) {
                                f2 x[4];
                                widen8(chunk(p, lc), x);
#pragma unroll
                                for (int m = 0; m < 4; ++m)
                                    acc[i][m] = add2(acc[i][m], mul_sep2(w2, x[m]));
                            }
                        }
                        release();
                    }
                    if (has_shared) {
                        const uint8_t *p = take();
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            if (FULL || lc < a.nchunks) add_bf16x8(acc[i], chunk(p, lc));
                        }
                        release();
                    }
                    // local BF16 rounding, then each chunk to its owner
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if (FULL || lc < a.nchunks) {
                            const uint4 z = round8(acc[i]);
                            if constexpr (REDUCE) {
                                // owner: the last CTA o whose slice starts at or before lc
                                const int o = ((lc + 1) * (int)cs + a.nchunks - 1) / a.nchunks - 1;
                                const int oc0 = (int)(((long long)o * a.nchunks) / (long long)cs);
                                const uint32_t dst = zb + (uint32_t)(r * zstride + (lc - oc0)) * 16u;
                                st_async_u4(mapa(dst, (uint32_t)o), z, mapa(zready, (uint32_t)o));
                            }
                            if ((Z_OUT || a.z_out != nullptr) && live)
                                *reinterpret_cast<uint4 *>(a.z_out + ((size_t)r * a.T + t) * H +
                                                           (size_t)lc * 8) = z;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.mempty0 + 8u * slot);
                if constexpr (REDUCE) {
                    if (!wait_phase<true, kDsmem, kOutline>(zready, (uint32_t)it & 1u, ctl)) live = false;
                    // rank-ordered sum of the R z rows over this CTA's slice,
                    // all from its own shared memory
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
                            widen8(zbuf[lc], s[i]);
                            // kept rolled: unrolled, this loop was a ninth of
                            // the shard-split kernel's code, and the smaller
                            // kernel is the faster one (C4 T=16 13.60 -> 13.37 us)
#pragma unroll 1
                            for (int rr = 1; rr < a.R; ++rr) add_bf16x8(s[i], zbuf[rr * zstride + lc]);
                        }
                    }
                }
            } else if constexpr (FIN) {
                if (!wait_phase<false, kPipe, kOutline>(sm.mfull0 + 8u * slot, ((uint32_t)it >> 1) & 1u, ctl))
                    live = false;
                const float *wrow = sm.mw + slot * kMaxMeta;
                for (int r = 0; r < a.R; ++r) {
                    f2 acc[CPT][4];
                    // slot 0: acc = w0 * x0
                    {
                        const float w0 = wrow[r * a.k];
                        const f2 w2 = f2_make(w0, w0);
                        const uint8_t *p = take();
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            f2 x[4] = {0ull, 0ull, 0ull, 0ull};
                            if ((FULL && !SPLITR) || lc < nch) widen8(chunk(p, lc), x);
#pragma unroll
                            for (int m = 0; m < 4; ++m) acc[i][m] = mul_sep2(w2, x[m]);
                        }
                        release();
                    }
                    // slots 1..k-1: acc = acc + wj * xj (two slots per iteration
                    // let the next copy's loads issue ahead of this one's adds)
#pragma unroll 2
                    for (int j = 1; j < a.k; ++j) {
                        const float wj = wrow[r * a.k + j];
                        const f2 w2 = f2_make(wj, wj);
                        const uint8_t *p = take();
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            if ((FULL && !SPLITR) || lc < nch) {
                                f2 x[4];
                                widen8(chunk(p, lc), x);
#pragma unroll
                                for (int m = 0; m < 4; ++m)
                                    acc[i][m] = add2(acc[i][m], mul_sep2(w2, x[m]));
                            }
                        }
                        release();
                    }
                    // shared-expert add
                    if (has_shared) {
                        const uint8_t *p = take();
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            if ((FULL && !SPLITR) || lc < nch) add_bf16x8(acc[i], chunk(p, lc));
                        }
                        release();
                    }
                    // local BF16 rounding, then the rank-ordered sum
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
                            const uint4 z = round8(acc[i]);
                            if ((Z_OUT || a.z_out != nullptr) && live)
                                *reinterpret_cast<uint4 *>(a.z_out + ((size_t)r * a.T + t) * H +
                                                           (size_t)(c0 + lc) * 8) = z;
                            if constexpr (REDUCE) {
                                if (r == 0)
                                    widen8(z, s[i]);
                                else
                                    add_bf16x8(s[i], z);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.mempty0 + 8u * slot);
            } else {
                // shard 0 initialises the sum, shards 1..R-1 add in rank order
                {
                    const uint8_t *p = take();
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) widen8(chunk(p, lc), s[i]);
                    }
                    release();
                }
                for (int r = 1; r < a.R; ++r) {
                    const uint8_t *p = take();
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) add_bf16x8(s[i], chunk(p, lc));
                    }
                    release();
                }
            }

            // ---- FP32 sum out (split path) or debug copy ----
            if constexpr (REDUCE && !SUM_IN) {
                if ((SUM_OUT || a.sum_out != nullptr) && live) {
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
                            f2 *dst = reinterpret_cast<f2 *>(a.sum_out + (size_t)t * H +
                                                             (size_t)(c0 + lc) * 8);
                            reinterpret_cast<ulonglong2 *>(dst)[0] = make_ulonglong2(s[i][0], s[i][1]);
                            reinterpret_cast<ulonglong2 *>(dst)[1] = make_ulonglong2(s[i][2], s[i][3]);
                        }
                    }
                }
            }

            // ---- norm-residual-norm ----
            if constexpr (RESNORM) {
                float ss1 = 0.f;
                if constexpr (POSTNORM) {
                    f2 S1 = 0ull, E1 = 0ull;
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
#pragma unroll
                            for (int m = 0; m < 4; ++m) acc_square2(S1, E1, s[i][m]);
                        }
                    }
                    ss1 = row_sum_squares<kOutline, SPLITR>(S1, E1, nred, sm, cs, q, NT, NW, warp, lane, tid, ctl, live);
                    if (TINY && needs_rescale(ss1)) {  // the same on every thread of the cluster
                        const int kx = rescale_exp(ss1);
                        const float up = pow2f(kx);
                        float Sb = 0.f, Eb = 0.f;
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            const int lc = tid + i * NT;
                            if ((FULL && !SPLITR) || lc < nch) {
#pragma unroll
                                for (int m = 0; m < 4; ++m) acc_square_scaled(Sb, Eb, s[i][m], up);
                            }
                        }
                        const float r = row_sum_squares<kOutline, SPLITR>(f2_make(Sb, 0.f), f2_make(Eb, 0.f), nred, sm, cs, q,
                                                        NT, NW, warp, lane, tid, ctl, live);
                        ss1 = mul_sep(mul_sep(r, pow2f(-kx)), pow2f(-kx));
                    }
                    const float r1 = rms_factor(ss1, a.H, a.eps);
                    const f2 r1x2 = f2_make(r1, r1);
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
                            f2 g[4];
                            gamma8(kGPost, i, g);
#pragma unroll
                            for (int m = 0; m < 4; ++m) s[i][m] = mul_sep2(mul2(s[i][m], r1x2), g[m]);
                        }
                    }
                }
                // residual add and write-back (s now holds y, or the sum itself)
                f2 S2 = 0ull, E2 = 0ull;
                {
                    const uint8_t *p = take();
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
                            add_bf16x8(s[i], chunk(p, lc));  // h = residual + y
#pragma unroll
                            for (int m = 0; m < 4; ++m) acc_square2(S2, E2, s[i][m]);
                            if (live)
                                *reinterpret_cast<uint4 *>(a.residual + (size_t)t * H +
                                                           (size_t)(c0 + lc) * 8) = round8(s[i]);
                        }
                    }
                    release();
                }
                float ss2 = row_sum_squares<kOutline, SPLITR>(S2, E2, nred, sm, cs, q, NT, NW, warp, lane, tid, ctl, live);
                if (TINY && needs_rescale(ss2)) {  // the same on every thread of the cluster
                    const int kx = rescale_exp(ss2);
                    const float up = pow2f(kx);
                    float Sb = 0.f, Eb = 0.f;
#pragma unroll
                    for (int i = 0; i < CPT; ++i) {
                        const int lc = tid + i * NT;
                        if ((FULL && !SPLITR) || lc < nch) {
#pragma unroll
                            for (int m = 0; m < 4; ++m) acc_square_scaled(Sb, Eb, s[i][m], up);
                        }
                    }
                    const float r = row_sum_squares<kOutline, SPLITR>(f2_make(Sb, 0.f), f2_make(Eb, 0.f), nred, sm, cs, q,
                                                    NT, NW, warp, lane, tid, ctl, live);
                    ss2 = mul_sep(mul_sep(r, pow2f(-kx)), pow2f(-kx));
                }
                const float r2 = rms_factor(ss2, a.H, a.eps);
                const f2 r2x2 = f2_make(r2, r2);
#pragma unroll
                for (int i = 0; i < CPT; ++i) {
                    const int lc = tid + i * NT;
                    if ((FULL && !SPLITR) || lc < nch) {
                        f2 g[4], o[4];
                        gamma8(kGPre, i, g);
#pragma unroll
                        for (int m = 0; m < 4; ++m) o[m] = mul2(mul2(s[i][m], r2x2), g[m]);
                        if (live)
                            *reinterpret_cast<uint4 *>(a.out + (size_t)t * H + (size_t)(c0 + lc) * 8) =
                                round8(o);
                    }
                }
                if (a.ss_out != nullptr && q == 0 && tid == 0 && live) {
                    a.ss_out[2 * (size_t)t] = ss1;
                    a.ss_out[2 * (size_t)t + 1] = ss2;
                }
            }
        }
    }
    // Release the next kernel in the stream only now: released at setup, its
    // CTAs would take SMs in the order this grid's SMs drain, which unbalances
    // rows when CTAs sharing an SM carry unequal loads (measured on GB300).
    griddep_launch_dependents();
    // The only accesses to another CTA's shared memory are remote stores (and
    // their byte counts) into the exchange slots, and every CTA waits for all
    // of those addressed to it before it gets here.  So a CTA leaves without a
    // cluster barrier (measured: 0.2 to 0.3 us less per call at few rows).
    // If one of its exchange waits gave up, stores from the other CTAs may
    // still be on their way: the threads that see it stay for the bounded
    // wait limit before leaving, and the CTA's shared memory lives as long as
    // they do.
    if (cs > 1 && (*(volatile int *)&s_abort & kAbortDsmem)) {
        const long long t0 = clock64();
        while (clock64() - t0 < kWaitLimitCycles) __nanosleep(1000);
    }
}

}  // namespace dev
}  // namespace bn
