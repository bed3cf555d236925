// kv_device.cuh -- device-side building blocks of the KV relocation library
// (sm_103a).  Row movement is HBM-bound: every row is read once and written
// once with 16-byte vector accesses; the rotary part is turned in fp32
// registers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kv_internal.h"

namespace kvr {

// ---------------------------------------------------------------------------
// 16-byte global accesses
// ---------------------------------------------------------------------------

// Streaming (evict-first) read and write of KV rows: each byte is touched once.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

// ---------------------------------------------------------------------------
// bf16 arithmetic helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool bf16_finite(uint32_t h) { return (h & 0x7F80u) != 0x7F80u; }

// Error-free sum: s + e == a + b exactly (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = a + b;
    float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Round the value hi + lo (|lo| at most half an fp32 ulp of hi) to the
// nearest bf16, ties to even.  hi alone decides unless it sits exactly on a
// bf16 tie; then the sign of lo says on which side the value lies.  NaN
// becomes the canonical quiet NaN 0x7FC0.
__device__ __forceinline__ uint32_t bf16_round(float hi, float lo)
{
    uint32_t u = __float_as_uint(hi);
    if ((u & 0x7F800000u) == 0x7F800000u)
        return (u & 0x007FFFFFu) ? 0x7FC0u : (u >> 16);
    uint32_t keep = u >> 16, low = u & 0xFFFFu;
    bool up;
    if (low != 0x8000u)
        up = low > 0x8000u;
    else if (lo != 0.0f)
        up = (__float_as_uint(lo) >> 31) == (u >> 31);
    else
        up = keep & 1u;
    return keep + (up ? 1u : 0u);
}

// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic.
typedef unsigned long long f2;

// bf16 pair (low half = first element) -> fp32 pair, exact.
__device__ __forceinline__ f2 f2_of_bf16x2(uint32_t w)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xFFFF0000u));
    return r;
}

__device__ __forceinline__ f2 f2_of_bits(uint32_t lo, uint32_t hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f2 f2_mul(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 f2_add(f2 a, f2 b)
{
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// fp32 pair -> bf16 pair, each rounded to nearest even (NaN stays NaN).
__device__ __forceinline__ uint32_t bf16x2_rne(f2 v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// True when either lane is NaN.
__device__ __forceinline__ bool f2_has_nan(f2 v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo != lo || hi != hi;
}

// ---------------------------------------------------------------------------
// The rotation R(δ) of one (x, y) = (x[j], x[j+d/2]) pair
// ---------------------------------------------------------------------------
//
// The δ-table stores, per (unit, frequency j), cos(δθ_j) = c1 + c2 and
// sin(δθ_j) = s1 + s2, formed in fp64; c1 and s1 carry at most 16
// significant bits, so with bf16 inputs (8 bits) the products x*c1 and y*s1
// are exact in fp32.  An error-free two-sum turns x*c1 - y*s1 into t + et
// exactly; the small c2/s2 terms (the next 24 bits of cos and sin) are
// added to et.  (hi, lo) then holds the rotated value to about 2^-38 of
// |x|+|y|, and one tie-aware rounding gives the bf16 nearest to it.

// The exact path: the rotated value to ~2^-38 of |x|+|y| as (hi, lo) and one
// tie-aware rounding.  `first` selects x*cos - y*sin (the lane holding the
// first half of the head) or x*sin + y*cos (second half); `add` is an fp32
// term (the rank-m patch, or 0) added before rounding.
static __device__ __noinline__ uint32_t rotate_one_exact(uint32_t xb, uint32_t yb, float4 cs, bool first,
                                                  float add)
{
    const float x = __uint_as_float(xb << 16), y = __uint_as_float(yb << 16);
    float hi, lo;
    if (bf16_finite(xb) && bf16_finite(yb)) {
        float p, q, u;
        if (first) {
            p = x * cs.x;    // exact
            q = -(y * cs.z); // exact
            u = fmaf(x, cs.y, -(y * cs.w));
        } else {
            p = x * cs.z;
            q = y * cs.x;
            u = fmaf(x, cs.w, y * cs.y);
        }
        float t, et;
        two_sum(p, q, t, et);
        if (fabsf(t) > 3.40282347e38f) {
            // x*c1 + y*s1 reaches the fp32 overflow threshold (inputs near
            // bf16's largest value): redo at half scale -- exact, the
            // operands are far from the subnormal range -- and double the
            // rounded result; beyond bf16's largest finite value the
            // doubling gives Inf, as rounding the fp64 value does.
            two_sum(0.5f * p, 0.5f * q, t, et);
            two_sum(t, et + 0.5f * u, hi, lo);
            float s, e;
            two_sum(hi, lo + 0.5f * add, s, e);
            const uint32_t r = bf16_round(s, e);
            return ((r & 0x7F80u) == 0x7F00u) ? ((r & 0x8000u) | 0x7F80u) : r + 0x80u;
        }
        two_sum(t, et + u, hi, lo);
    } else {
        // Inf / NaN inputs: plain IEEE arithmetic, as the fp64 definition does
        const float c = cs.x + cs.y, s = cs.z + cs.w;
        hi = first ? (x * c - y * s) : (x * s + y * c);
        lo = 0.0f;
    }
    float s, e;
    two_sum(hi, lo + add, s, e);
    return bf16_round(s, e);
}

// Same result, cheaply: with exact leading products (inputs above fp32's
// subnormal range), t + (u + add) is the rotated value to within about
// 2^-23 (|x| + |y| + |add|), so its round-to-nearest-even is already the
// correctly rounded bf16 unless a bf16 rounding boundary lies near it (the
// interval test below), or it is not finite.  Those rare cases (about one
// value in 10^4) take the exact path.
__device__ __forceinline__ uint32_t rotate_one(uint32_t xb, uint32_t yb, float4 cs, bool first,
                                               float add)
{
    const float x = __uint_as_float(xb << 16), y = __uint_as_float(yb << 16);
    float t, u;
    if (first) {
        t = fmaf(x, cs.x, -(y * cs.z));
        u = fmaf(x, cs.y, -(y * cs.w));
    } else {
        t = fmaf(x, cs.z, y * cs.x);
        u = fmaf(x, cs.w, y * cs.y);
    }
    const float s = t + (u + add);
    // s is within 2^-23 (|x| + |y| + |add|)(1 + 2^-15) of the exact value
    // (two roundings of terms no larger than |x| + |y| + |add|, plus the
    // small c2/s2 terms); the ends s +- 2^-22 (|x| + |y| + |add|) lie beyond
    // that distance even after their own rounding, so if both ends round to
    // the same bf16, so does the exact value (rounding is monotone).  This
    // also covers cancellation.
    const float r = 2.384185791015625e-7f * (fabsf(x) + fabsf(y) + fabsf(add)); // 2^-22
    uint32_t ends;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(ends) : "f"(s + r), "f"(s - r));
    if (((ends ^ (ends >> 16)) & 0xFFFFu) != 0u || !(fabsf(s) <= 3.40282347e38f))
        return rotate_one_exact(xb, yb, cs, first, add);
    return ends & 0xFFFFu;
}

// Patched values are held to 1 bf16 ulp (the fp32 patch sum carries its
// own ~1e-10 error), so they take a shorter path than the exact rotation.

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16, round to nearest even; NaN -> 0x7FC0.
__device__ __forceinline__ uint32_t bf16_rne(float f)
{
    const uint32_t u = __float_as_uint(f);
    const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return ((u & 0x7FFFFFFFu) > 0x7F800000u) ? 0x7FC0u : r;
}

// rnd(R(δ)·(x, y) + add) for this lane's half, with two FMAs per product
// (cos = c1 + c2, sin = s1 + s2 from the table).
__device__ __forceinline__ uint32_t rotate_add_fast(uint32_t xb, uint32_t yb, float4 cs,
                                                    bool first, float add)
{
    const float x = __uint_as_float(xb << 16), y = __uint_as_float(yb << 16);
    if (!(bf16_finite(xb) && bf16_finite(yb))) {
        // Inf / NaN inputs: plain IEEE arithmetic, as the fp64 definition does
        const float c = cs.x + cs.y, s = cs.z + cs.w;
        return bf16_rne((first ? (x * c - y * s) : (x * s + y * c)) + add);
    }
    float t, u;
    if (first) {
        t = fmaf(x, cs.x, -(y * cs.z));
        u = fmaf(x, cs.y, -(y * cs.w));
    } else {
        t = fmaf(x, cs.z, y * cs.x);
        u = fmaf(x, cs.w, y * cs.y);
    }
    return bf16_rne(t + (u + add));
}

// x + add, rounded once (patch on a verbatim value).
__device__ __forceinline__ uint32_t add_round(uint32_t xb, float add)
{
    const float x = __uint_as_float(xb << 16);
    float s, e;
    two_sum(x, add, s, e);
    return bf16_round(s, e);
}

// Rotate one 16-byte vector (8 bf16) of a head.  `mine` is this lane's
// vector, `other` its partner's (the same 8 frequencies in the other half),
// `first` tells whether `mine` lies in the first half.  The table entry of
// element e is cs[e * cs_step]; add[8] is the patch term (or zeros).
__device__ __forceinline__ uint4 rotate_vec(uint4 mine, uint4 other, bool first,
                                            const float4 *cs, int cs_step, const float *add)
{
    const uint32_t m[4] = {mine.x, mine.y, mine.z, mine.w};
    const uint32_t o[4] = {other.x, other.y, other.z, other.w};
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t xw = first ? m[k] : o[k];
        const uint32_t yw = first ? o[k] : m[k];
        const uint32_t r0 =
            rotate_one(xw & 0xFFFFu, yw & 0xFFFFu, cs[(2 * k) * cs_step], first, add[2 * k]);
        const uint32_t r1 =
            rotate_one(xw >> 16, yw >> 16, cs[(2 * k + 1) * cs_step], first, add[2 * k + 1]);
        out[k] = r0 | (r1 << 16);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Pair-packed cos/sin (rows without a patch term).  For word k of a vector
// (its elements e0 = 2k and e1 = 2k + 1) the shared-memory row holds
//   cs[(2k)   * step] = (c1[e0], c1[e1], s1[e0], s1[e1])
//   cs[(2k+1) * step] = (c2[e0], c2[e1], s2[e0], s2[e1])
// so each 16-byte load yields the two register pairs of an f32x2 operand.
// Each lane forms mine*cos + partner*(±sin): with the partner negated in
// the first half of the head that is x cos - y sin, in the second half
// y cos + x sin -- the same exact products as rotate_one, two at a time.

// The exact path for one word.  a, b are the word's two table entries; mw,
// ow this lane's and the partner's words.
__device__ __forceinline__ uint32_t rotate_word_exact(uint32_t mw, uint32_t ow, bool first,
                                                      float4 a, float4 b)
{
    const uint32_t xw = first ? mw : ow;
    const uint32_t yw = first ? ow : mw;
    const uint32_t r0 = rotate_one_exact(xw & 0xFFFFu, yw & 0xFFFFu,
                                         make_float4(a.x, b.x, a.z, b.z), first, 0.0f);
    const uint32_t r1 = rotate_one_exact(xw >> 16, yw >> 16,
                                         make_float4(a.y, b.y, a.w, b.w), first, 0.0f);
    return r0 | (r1 << 16);
}

// Redo the words of a vector whose fast results failed the interval test
// (rare: a result within the test's distance of a bf16 rounding boundary, or
// not finite); `bad` is nonzero for those words.
static __device__ __noinline__ uint4 fix_vec_packed(uint4 out, uint4 bad, uint4 mine, uint4 other,
                                                    bool first, const float4 *cs, int step)
{
    uint32_t r[4] = {out.x, out.y, out.z, out.w};
    const uint32_t b[4] = {bad.x, bad.y, bad.z, bad.w};
    const uint32_t m[4] = {mine.x, mine.y, mine.z, mine.w};
    const uint32_t o[4] = {other.x, other.y, other.z, other.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (b[k])
            r[k] = rotate_word_exact(m[k], o[k], first, cs[(2 * k) * step],
                                     cs[(2 * k + 1) * step]);
    return make_uint4(r[0], r[1], r[2], r[3]);
}

__device__ __forceinline__ f2 f2_abs(f2 v) { return v & 0x7FFFFFFF7FFFFFFFull; }

// Rotate one 16-byte vector with f32x2 arithmetic and the same interval
// test as rotate_one, applied to both elements of a word at once: the ends
// s ± 2^-22 (|x| + |y|) are rounded as one bf16 pair each; if the pairs
// agree and are finite the word is the correctly rounded result.  One branch
// per vector, so the four words' arithmetic interleaves.
__device__ __forceinline__ uint4 rotate_vec_packed(uint4 mine, uint4 other, bool first,
                                                   const float4 *cs, int step)
{
    const uint32_t m[4] = {mine.x, mine.y, mine.z, mine.w};
    const uint32_t o[4] = {other.x, other.y, other.z, other.w};
    const uint32_t sgn = first ? 0x80008000u : 0u;
    const f2 kUp = 0x3480000034800000ull;   // (2^-22, 2^-22)
    const f2 kDn = 0xB4800000B4800000ull;   // (-2^-22, -2^-22)
    uint32_t out[4], bad[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 a = cs[(2 * k) * step], b = cs[(2 * k + 1) * step];
        const f2 c1 = f2_of_bits(__float_as_uint(a.x), __float_as_uint(a.y));
        const f2 s1 = f2_of_bits(__float_as_uint(a.z), __float_as_uint(a.w));
        const f2 c2 = f2_of_bits(__float_as_uint(b.x), __float_as_uint(b.y));
        const f2 s2 = f2_of_bits(__float_as_uint(b.z), __float_as_uint(b.w));
        const f2 x = f2_of_bf16x2(m[k]);
        const f2 y = f2_of_bf16x2(o[k] ^ sgn);
        const f2 t = f2_fma(x, c1, f2_mul(y, s1));   // one rounding of exact products
        const f2 u = f2_fma(x, c2, f2_mul(y, s2));   // the next 24 bits of cos / sin
        const f2 s = f2_add(t, u);
        const f2 mag = f2_add(f2_abs(x), f2_abs(y));
        const uint32_t hi = bf16x2_rne(f2_fma(mag, kUp, s));
        const uint32_t lo = bf16x2_rne(f2_fma(mag, kDn, s));
        // disagreement, or an Inf / NaN half (exponent field all ones)
        bad[k] = (hi ^ lo) | (((hi & 0x7FFF7FFFu) + 0x00800080u) & 0x80008000u);
        out[k] = hi;
    }
    const uint4 res = make_uint4(out[0], out[1], out[2], out[3]);
    if ((bad[0] | bad[1]) | (bad[2] | bad[3]))
        return fix_vec_packed(res, make_uint4(bad[0], bad[1], bad[2], bad[3]), mine, other, first,
                              cs, step);
    return res;
}

__device__ __forceinline__ uint4 add_vec(uint4 x, const float *add)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        out[k] = add_round(w[k] & 0xFFFFu, add[2 * k]) |
                 (add_round(w[k] >> 16, add[2 * k + 1]) << 16);
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ uint4 shfl_xor_u4(uint4 v, int mask)
{
    v.x = __shfl_xor_sync(0xFFFFFFFFu, v.x, mask);
    v.y = __shfl_xor_sync(0xFFFFFFFFu, v.y, mask);
    v.z = __shfl_xor_sync(0xFFFFFFFFu, v.z, mask);
    v.w = __shfl_xor_sync(0xFFFFFFFFu, v.w, mask);
    return v;
}

// ---------------------------------------------------------------------------
// Status word and bounded waits
// ---------------------------------------------------------------------------

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_status(uint32_t *status, uint32_t code)
{
    atomicCAS(status, 0u, code);
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Named barrier `id` over `count` threads of the block: bar_arrive signals
// (and orders the caller's earlier memory accesses before the waiters'
// later ones) without waiting; bar_wait_all waits for the phase to complete.
__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t count)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_wait_all(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Spin until *flag != 0, for at most limit_ns of wall time and at most a
// fixed number of polls (the poll cap bounds the wait even if the timer
// misbehaves).  Returns false if the wait ran out.
static __device__ __noinline__ bool wait_flag(const uint32_t *flag, int64_t limit_ns)
{
    const uint64_t t0 = global_ns();
    const uint64_t max_polls = (uint64_t)limit_ns / 16u + 4096u;
    unsigned sleep_ns = 32;
    for (uint64_t it = 0; it < max_polls; ++it) {
        if (ld_acquire(flag) != 0u)
            return true;
        if ((int64_t)(global_ns() - t0) > limit_ns)
            return false;
        __nanosleep(sleep_ns);
        if (sleep_ns < 2048)
            sleep_ns <<= 1;
    }
    return ld_acquire(flag) != 0u;
}

// Spin until *counter >= want, bounded as wait_flag; returns the last value
// read (>= want on success).
static __device__ __noinline__ uint32_t wait_count(const uint32_t *counter, uint32_t want,
                                                   int64_t limit_ns)
{
    const uint64_t t0 = global_ns();
    const uint64_t max_polls = (uint64_t)limit_ns / 16u + 4096u;
    unsigned sleep_ns = 32;
    uint32_t v = 0;
    for (uint64_t it = 0; it < max_polls; ++it) {
        v = ld_acquire(counter);
        if (v >= want)
            return v;
        if ((int64_t)(global_ns() - t0) > limit_ns)
            return v;
        // the awaited tile is usually a fraction of a microsecond away: a
        // short backoff keeps the detection delay small
        __nanosleep(sleep_ns);
        if (sleep_ns < 256)
            sleep_ns <<= 1;
    }
    return ld_acquire(counter);
}

// ---------------------------------------------------------------------------
// δ-table entry: cos/sin of δ·θ_j in fp64, stored as two-part fp32
// ---------------------------------------------------------------------------

// Keep the 16 leading significant bits of a double (truncation).
__device__ __forceinline__ double lead16(double x)
{
    return __longlong_as_double(__double_as_longlong(x) & ~((1ll << 37) - 1));
}

// (c1, c2, s1, s2) with cos(δθ_j) = c1 + c2 and sin(δθ_j) = s1 + s2, the
// angle and its cosine / sine formed in fp64, θ_j = base^(-2j/d); c1 and s1
// keep at most 16 significant bits, so their products with bf16 values are
// exact in fp32.
__device__ __forceinline__ float4 delta_entry(int32_t delta, int j, int head_dim, double base)
{
    const double theta = pow(base, -2.0 * (double)j / (double)head_dim);
    const double a = (double)delta * theta;
    double s, c;
    sincos(a, &s, &c);
    const double c1 = lead16(c), s1 = lead16(s);
    return make_float4((float)c1, (float)(c - c1), (float)s1, (float)(s - s1));
}

// The same entry behind a call boundary, for kernels that form their table
// row in a prologue: the fp64 library code then does not weigh on the
// registers of the kernel's main loop.
static __device__ __noinline__ float4 delta_entry_call(int32_t delta, int j, int head_dim,
                                                       double base)
{
    return delta_entry(delta, j, head_dim, base);
}

// Physical slot of logical position pos in a block-table row, or -1 when
// the position or the block id falls outside the table or the pool.
__device__ __forceinline__ int64_t slot_of(const int32_t *bt_row, int32_t max_blocks,
                                           int32_t block, int64_t num_blocks, int64_t pos)
{
    if (pos < 0)
        return -1;
    const int64_t b = pos / block;
    if (b >= max_blocks)
        return -1;
    const int64_t blk = bt_row[b];
    if (blk < 0 || blk >= num_blocks)
        return -1;
    return blk * block + pos % block;
}

} // namespace kvr
