// kv_cdc.cu -- content-defined chunking of token streams on the GPU.
//
// Irminsul §2.2 (content hash keying with CDC): a Gear rolling hash over
// windows of 64 tokens ends a chunk where it falls below a threshold, so the
// boundaries follow the content; each chunk is named by its xxHash64
// fingerprint; the fixed-window fallback (S1) names 128-token windows.
//
//   h(i) = 2 h(i-1) + G(x_i) mod 2^64, h = 0 before a stream's first token,
//   G(x) = output number x of SplitMix64 seeded with gear_seed,
//   a chunk ends after token i when h(i) < threshold, and at its stream's end,
//   fingerprint = XXH64 of the chunk's token ids as 4-byte little-endian words.
//
// Kernels of one call:
//   1. cdc_flags_kernel: a block owns 8192 positions and stages G for them and
//      the 64 before them in shared memory (coalesced), with a bit mask of the
//      stream starts among them.  The Gear recurrence
//      is linear, so a thread first hashes its 32 positions from zero (the
//      run's own part), then takes the hash entering its run from the two
//      runs before it -- h(a-1) = H(run-1) + 2^32 H(run-2) mod 2^64, the
//      runs further back are shifted out -- and rolls its run again, keeping
//      one bit per position where a chunk ends; per-block counts and the last
//      chunk end of the block.
//   2. cdc_scan_kernel: one block turns the counts into offsets (and the
//      total) and the last ends into "where the first chunk of each block
//      starts".
//   3. cdc_emit_kernel: a block stages its tile's tokens and the 1024 before
//      them; each set bit becomes a chunk end, in stream order; a chunk under
//      64 tokens is hashed by the thread owning its end, a longer one by four
//      lanes, one XXH64 accumulator each (shared memory, global memory for a
//      part that starts further back).
// kv_fingerprint runs fingerprint_kernel: one thread per range.
#include "kv_device.cuh"
#include "kv_launch.h"

namespace kvr {
namespace {

constexpr int kThreadsCdc = 256;
constexpr int kRun = 32;                         // positions per thread
constexpr int kTileCdc = kThreadsCdc * kRun;     // positions per block
constexpr int kHalo = 2 * kRun;                  // the two runs before a tile: the 64-token window
constexpr int kStageEntries = kTileCdc + kHalo;
constexpr int kLookback = 1024;                  // tokens before a tile staged for hashing
// one spare entry per 32, so the lanes of a warp, 32 positions apart, hit
// different banks
constexpr int kStagePadded = kStageEntries + kStageEntries / 32 + 1;

__device__ __forceinline__ int staged(int r) { return r + (r >> 5); }

// Output number x of SplitMix64 seeded with `seed` (Steele, Lea and Flood,
// OOPSLA 2014): the state after x + 1 golden-ratio steps, then the mix.
__device__ __forceinline__ uint64_t gear_value(uint64_t seed, uint32_t x)
{
    uint64_t z = seed + ((uint64_t)x + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// ---- XXH64 (Collet's published algorithm) over 4-byte token words ----

constexpr uint64_t kP1 = 0x9E3779B185EBCA87ull;
constexpr uint64_t kP2 = 0xC2B2AE3D27D4EB4Full;
constexpr uint64_t kP3 = 0x165667B19E3779F9ull;
constexpr uint64_t kP4 = 0x85EBCA77C2B2AE63ull;
constexpr uint64_t kP5 = 0x27D4EB2F165667C5ull;

__device__ __forceinline__ uint64_t rotl(uint64_t v, int r) { return (v << r) | (v >> (64 - r)); }

__device__ __forceinline__ uint64_t xround(uint64_t acc, uint64_t lane)
{
    return rotl(acc + lane * kP2, 31) * kP1;
}

// Token words from global memory.
struct GlobalTokens {
    const int32_t *t;
    __device__ __forceinline__ uint32_t operator()(int64_t i) const { return (uint32_t)__ldg(t + i); }
};

// Token words from a staged range [lo, hi) of shared memory, global memory
// outside it.
struct StagedTokens {
    const uint32_t *s;
    int64_t lo, hi;
    const int32_t *t;
    __device__ __forceinline__ uint32_t operator()(int64_t i) const
    {
        return (i >= lo && i < hi) ? s[i - lo] : (uint32_t)__ldg(t + i);
    }
};

// Token words from shared memory, indexed from a chunk's first token.
struct SharedTokens {
    const uint32_t *c;
    __device__ __forceinline__ uint32_t operator()(int64_t i) const { return c[i]; }
};

// Eight bytes = tokens i, i+1 as little-endian words.
template <class F>
__device__ __forceinline__ uint64_t lane8(const F &tok, int64_t i)
{
    return (uint64_t)tok(i) | ((uint64_t)tok(i + 1) << 32);
}

// XXH64 of tokens [a, b): 32-byte stripes (8 tokens) into four accumulators,
// then 8-byte pieces, then at most one 4-byte word, then the avalanche.
template <class F>
__device__ __forceinline__ uint64_t xxh64_tokens(const F &tok, int64_t a, int64_t b, uint64_t seed)
{
    const int64_t n = b - a;
    int64_t i = a;
    uint64_t acc;
    if (n >= 8) {
        uint64_t v1 = seed + kP1 + kP2, v2 = seed + kP2, v3 = seed, v4 = seed - kP1;
        for (; i + 8 <= b; i += 8) {
            v1 = xround(v1, lane8(tok, i));
            v2 = xround(v2, lane8(tok, i + 2));
            v3 = xround(v3, lane8(tok, i + 4));
            v4 = xround(v4, lane8(tok, i + 6));
        }
        acc = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
        acc = (acc ^ xround(0, v1)) * kP1 + kP4;
        acc = (acc ^ xround(0, v2)) * kP1 + kP4;
        acc = (acc ^ xround(0, v3)) * kP1 + kP4;
        acc = (acc ^ xround(0, v4)) * kP1 + kP4;
    } else {
        acc = seed + kP5;
    }
    acc += (uint64_t)(n * 4);
    for (; i + 2 <= b; i += 2) {
        acc ^= xround(0, lane8(tok, i));
        acc = rotl(acc, 27) * kP1 + kP4;
    }
    if (i < b) { // one 4-byte word left (token counts leave no single bytes)
        acc ^= (uint64_t)tok(i) * kP1;
        acc = rotl(acc, 23) * kP2 + kP3;
    }
    acc ^= acc >> 33;
    acc *= kP2;
    acc ^= acc >> 29;
    acc *= kP3;
    acc ^= acc >> 32;
    return acc;
}

// Stream starts at positions lo .. hi (and the end of all tokens, which
// closes the last stream) as bits q - base of a shared-memory mask: a
// block-parallel search for the first offset in range, then a block-strided
// walk over the offsets in range.
__device__ __forceinline__ void stage_starts(const CdcParams &p, int64_t base, int64_t lo,
                                             int64_t hi, uint32_t *s_start, int words,
                                             int *s_found)
{
    const int tid = threadIdx.x;
    for (int w = tid; w < words; w += blockDim.x)
        s_start[w] = 0u;
    // first s in [0, num_streams] with stream_off[s] >= lo: each round samples
    // the candidate interval at kThreadsCdc points (one load per thread), so
    // a few rounds replace a chain of dependent loads
    int a = 0, b = p.num_streams;
    while (a < b) {
        const int step = (b - a + kThreadsCdc) / kThreadsCdc; // ceil((b - a + 1) / threads)
        if (tid == 0)
            *s_found = b;
        __syncthreads();
        const int64_t idx = (int64_t)a + (int64_t)tid * step;
        if (idx <= b && p.stream_off[idx] >= lo)
            atomicMin(s_found, (int)idx);
        __syncthreads();
        const int f = *s_found;
        __syncthreads();
        a = max(a, f - step + 1); // the sample before f lies below lo
        b = f;
    }
    for (int s = a + tid; s <= p.num_streams; s += blockDim.x) {
        const int64_t o = p.stream_off[s];
        if (o > hi)
            break;
        if (o >= lo)
            atomicOr(&s_start[(o - base) >> 5], 1u << ((o - base) & 31));
    }
}

// Hash of the (up to) 32-position run at tile offset r0 (a multiple of 32,
// so its start bits are word r0/32 of the mask) from zero, cut at every
// stream start in it; `started` tells whether a stream starts inside the run
// (then nothing before the run reaches its end).
__device__ __forceinline__ uint64_t run_hash(const uint64_t *s_g, const uint32_t *s_start, int r0,
                                             int n, bool &started)
{
    const uint64_t *g = s_g + staged(r0); // positions r0 .. r0+31 are contiguous
    const uint32_t sw = s_start[r0 >> 5];
    uint64_t h = 0;
    if (n == kRun && sw == 0u) { // a whole run inside one stream (the common case)
#pragma unroll
        for (int j = 0; j < kRun; ++j)
            h = (h << 1) + g[j];
        started = false;
        return h;
    }
#pragma unroll
    for (int j = 0; j < kRun; ++j) {
        if (j < n) {
            if ((sw >> j) & 1u)
                h = 0;
            h = 2u * h + g[j];
        }
    }
    started = (sw & (n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u))) != 0u;
    return h;
}

__global__ void __launch_bounds__(kThreadsCdc) cdc_flags_kernel(const __grid_constant__ CdcParams p)
{
    extern __shared__ uint64_t s_g[];
    __shared__ uint32_t s_start[(kStageEntries + 1 + 31) / 32];
    __shared__ uint64_t s_run[kThreadsCdc + 2];   // run hashes; [0], [1] = the halo runs
    __shared__ int32_t s_started[kThreadsCdc + 2];
    __shared__ int64_t s_warp[kThreadsCdc / 32];
    __shared__ int64_t s_wlast[kThreadsCdc / 32];
    __shared__ int s_found;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t tile0 = (int64_t)blockIdx.x * kTileCdc;
    const int64_t lo = tile0 - kHalo;                 // offset r = q - lo
    const int64_t hi = min(tile0 + kTileCdc, p.total);

    if (blockIdx.x == 0 && tid == 0) {
        if (p.stream_off[0] != 0 || p.stream_off[p.num_streams] != p.total)
            set_status(p.status, kStatusOutOfRange);
    }
    // the tile's loads in flight in two batches, then their Gear values
    constexpr int kPer = (kStageEntries + kThreadsCdc - 1) / kThreadsCdc;
    constexpr int kBatch = (kPer + 1) / 2;
#pragma unroll
    for (int k0 = 0; k0 < kPer; k0 += kBatch) {
        uint32_t x[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int64_t q = lo + tid + (k0 + k) * kThreadsCdc;
            x[k] = (k0 + k < kPer && q >= 0 && q < hi) ? (uint32_t)__ldg(p.tokens + q) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int64_t q = lo + tid + (k0 + k) * kThreadsCdc;
            if (k0 + k < kPer && q >= 0 && q < hi)
                s_g[staged(tid + (k0 + k) * kThreadsCdc)] = gear_value(p.gear_seed, x[k]);
        }
    }
    // positions lo .. hi, both ends included: a start at hi ends the stream before it
    stage_starts(p, lo, max(lo, (int64_t)0), hi, s_start, (kStageEntries + 1 + 31) / 32,
                 &s_found);
    __syncthreads();

    // pass 1: every run's own hash (threads 0 and 1 also take the halo runs)
    const int64_t p0 = tile0 + (int64_t)tid * kRun;
    const int r0 = kHalo + tid * kRun;
    const int n = (int)max((int64_t)0, min((int64_t)kRun, p.total - p0));
    bool st;
    s_run[tid + 2] = run_hash(s_g, s_start, r0, n, st);
    s_started[tid + 2] = st;
    if (tid < 2) {
        s_run[tid] = lo < 0 ? 0ull : run_hash(s_g, s_start, tid * kRun, kRun, st);
        s_started[tid] = lo < 0 ? 1 : st;
    }
    __syncthreads();

    // pass 2: the hash entering my run, then my run again with the flags
    uint32_t flags = 0;
    int64_t last_end = -1;
    if (n > 0) {
        uint64_t h = s_run[tid + 1] + (s_started[tid + 1] ? 0ull : (s_run[tid] << 32));
        const uint64_t *g = s_g + staged(r0);
        const uint32_t sw = s_start[r0 >> 5];
        // a chunk also ends where the next position starts a stream
        const uint32_t ends = (sw >> 1) | ((s_start[(r0 >> 5) + 1] & 1u) << 31);
        if (n == kRun && sw == 0u) { // the common case: no stream starts in the run
#pragma unroll
            for (int j = 0; j < kRun; ++j) {
                h = (h << 1) + g[j];
                flags |= (uint32_t)(h < p.threshold) << j;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kRun; ++j) {
                if (j < n) {
                    if ((sw >> j) & 1u)
                        h = 0;
                    h = (h << 1) + g[j];
                    if (h < p.threshold)
                        flags |= 1u << j;
                }
            }
        }
        flags |= ends & (n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u));
        if (flags)
            last_end = p0 + (31 - __clz(flags)) + 1;
    }
    p.flags[(int64_t)blockIdx.x * kThreadsCdc + tid] = flags;

    int64_t c = __popc(flags), m = last_end;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    }
    if (lane == 0) {
        s_warp[warp] = c;
        s_wlast[warp] = m;
    }
    __syncthreads();
    if (tid == 0) {
        int64_t t = 0, l = -1;
#pragma unroll
        for (int w = 0; w < kThreadsCdc / 32; ++w) {
            t += s_warp[w];
            l = max(l, s_wlast[w]);
        }
        p.block_count[blockIdx.x] = t;
        p.block_last[blockIdx.x] = l;
    }
}

// One block of 1024 threads: exclusive sum of the per-block counts (chunk
// offsets, and the total) and exclusive running maximum of the per-block
// last chunk ends (where each block's first chunk starts; 0 for none).
__global__ void __launch_bounds__(1024) cdc_scan_kernel(const __grid_constant__ CdcParams p)
{
    __shared__ int64_t s_sum[1024];
    __shared__ int64_t s_max[1024];
    const int tid = threadIdx.x;
    const int per = (p.blocks + 1023) / 1024;
    const int b0 = min(tid * per, p.blocks), b1 = min(b0 + per, p.blocks);
    int64_t sum = 0, mx = 0;
    for (int b = b0; b < b1; ++b) {
        sum += p.block_count[b];
        mx = max(mx, p.block_last[b]);
    }
    s_sum[tid] = sum;
    s_max[tid] = mx;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) { // inclusive Hillis-Steele scans
        const int64_t v = tid >= o ? s_sum[tid - o] : 0;
        const int64_t w = tid >= o ? s_max[tid - o] : 0;
        __syncthreads();
        s_sum[tid] += v;
        s_max[tid] = max(s_max[tid], w);
        __syncthreads();
    }
    int64_t run = s_sum[tid] - sum;
    int64_t prev = tid > 0 ? s_max[tid - 1] : 0;
    for (int b = b0; b < b1; ++b) {
        p.block_off[b] = run;
        p.block_prev_end[b] = prev;
        run += p.block_count[b];
        prev = max(prev, p.block_last[b]);
    }
    if (tid == 1023) {
        *p.num_chunks = s_sum[1023];
        if (s_sum[1023] > p.max_chunks)
            set_status(p.status, kStatusCapacity);
    }
}

// Chunks of at least kLongChunk tokens are hashed by four lanes, one XXH64
// accumulator each; at most kTileCdc / kLongChunk + 1 of them end in a tile
// (they are disjoint and only the first can start before it).
constexpr int kLongChunk = 64;
constexpr int kMaxLong = kTileCdc / kLongChunk + 1;

// Every set flag bit becomes a chunk end (exclusive, a global token offset)
// and its fingerprint: short chunks are hashed by the lane owning the end,
// long ones by a quad of lanes (accumulator a over the 8-byte lane a of every
// 32-byte stripe; lane 0 of the quad merges and hashes the tail).  A chunk
// starts at the previous end: the owner's previous bit, an earlier thread's
// last bit, or the block's entry from the scan.
__global__ void __launch_bounds__(kThreadsCdc) cdc_emit_kernel(const __grid_constant__ CdcParams p)
{
    extern __shared__ uint32_t s_tok[];
    __shared__ int64_t s_wsum[kThreadsCdc / 32];
    __shared__ int64_t s_wmax[kThreadsCdc / 32];
    __shared__ int64_t s_la[kMaxLong], s_lb[kMaxLong], s_lk[kMaxLong];
    __shared__ int16_t s_order[kMaxLong]; // long chunks, longest first
    __shared__ int s_nlong;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t tile0 = (int64_t)blockIdx.x * kTileCdc;
    const int64_t lo = max(tile0 - kLookback, (int64_t)0);
    const int64_t hi = min(tile0 + kTileCdc, p.total);
    {   // every load of the staged range in flight at once
        constexpr int kPer = (kTileCdc + kLookback + kThreadsCdc - 1) / kThreadsCdc;
        uint32_t x[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int64_t q = lo + tid + k * kThreadsCdc;
            x[k] = q < hi ? (uint32_t)__ldg(p.tokens + q) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            if (lo + tid + k * kThreadsCdc < hi)
                s_tok[tid + k * kThreadsCdc] = x[k];
    }
    if (tid == 0)
        s_nlong = 0;

    const uint32_t flags = p.flags[(int64_t)blockIdx.x * kThreadsCdc + tid];
    const int64_t p0 = tile0 + (int64_t)tid * kRun;
    const int c = __popc(flags);
    int incl = c;
    int64_t mx = flags ? p0 + (31 - __clz(flags)) + 1 : 0; // my last chunk end
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        const int64_t w = __shfl_up_sync(0xFFFFFFFFu, mx, o);
        if (lane >= o) {
            incl += v;
            mx = max(mx, w);
        }
    }
    const int64_t below = __shfl_up_sync(0xFFFFFFFFu, mx, 1); // the lanes below me
    if (lane == 31) {
        s_wsum[warp] = incl;
        s_wmax[warp] = mx;
    }
    __syncthreads(); // also: the tokens are staged, s_nlong is 0
    int64_t k = p.block_off[blockIdx.x];
    int64_t prev = p.block_prev_end[blockIdx.x];
    for (int w = 0; w < warp; ++w) {
        k += s_wsum[w];
        prev = max(prev, s_wmax[w]);
    }
    if (lane > 0)
        prev = max(prev, below);
    k += incl - c;
    const StagedTokens tok{s_tok, lo, hi, p.tokens};
    uint32_t f = flags;
    while (f) {
        const int j = __ffs(f) - 1;
        f &= f - 1;
        const int64_t e = p0 + j + 1;
        if (k < p.max_chunks) {
            p.chunk_end[k] = e;
            if (e - prev < kLongChunk) {
                p.fingerprint[k] = prev >= lo
                    ? xxh64_tokens(SharedTokens{s_tok + (prev - lo)}, 0, e - prev, p.fp_seed)
                    : xxh64_tokens(tok, prev, e, p.fp_seed);
            } else {
                const int i = atomicAdd(&s_nlong, 1);
                if (i < kMaxLong) {
                    s_la[i] = prev;
                    s_lb[i] = e;
                    s_lk[i] = k;
                }
            }
        }
        prev = e;
        ++k;
    }
    __syncthreads();

    // long chunks, longest first, so that the quads of a warp (which wait for
    // one another) get chunks of similar length; quad q takes the q-th, the
    // (q + 64)-th, ... of them
    const int nlong = min(s_nlong, kMaxLong);
    if (tid < nlong) {
        const int64_t len = s_lb[tid] - s_la[tid];
        int rank = 0;
        for (int j = 0; j < nlong; ++j) {
            const int64_t lj = s_lb[j] - s_la[j];
            rank += (lj > len) || (lj == len && j < tid);
        }
        s_order[rank] = (int16_t)tid;
    }
    __syncthreads();
    const int quad = tid >> 2, a = tid & 3;
    const int rounds = (nlong + kThreadsCdc / 4 - 1) / (kThreadsCdc / 4);
    for (int r = 0; r < rounds; ++r) {
        const int ri = quad + r * (kThreadsCdc / 4);
        const bool mine = ri < nlong;
        const int i = mine ? s_order[ri] : 0;
        const int64_t ca = mine ? s_la[i] : 0, cb = mine ? s_lb[i] : 0;
        const uint64_t seed = p.fp_seed;
        uint64_t v = a == 0 ? seed + kP1 + kP2 : a == 1 ? seed + kP2 : a == 2 ? seed : seed - kP1;
        int64_t q = ca;
        if (mine) {
            if (ca >= lo) { // the whole chunk is staged: 32-bit offsets into shared memory
                const uint32_t *cw = s_tok + (int)(ca - lo) + 2 * a;
                const int m8 = (int)((cb - ca) >> 3);
                for (int t = 0; t < m8; ++t)
                    v = xround(v, (uint64_t)cw[8 * t] | ((uint64_t)cw[8 * t + 1] << 32));
                q = ca + 8 * (int64_t)m8;
            } else {
                for (; q + 8 <= cb; q += 8)
                    v = xround(v, lane8(tok, q + 2 * a));
            }
        }
        // lanes 1..3 of the quad hand their accumulators to lane 0
        const uint64_t v2 = __shfl_down_sync(0xFFFFFFFFu, v, 1);
        const uint64_t v3 = __shfl_down_sync(0xFFFFFFFFu, v, 2);
        const uint64_t v4 = __shfl_down_sync(0xFFFFFFFFu, v, 3);
        if (mine && a == 0) {
            uint64_t acc = rotl(v, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
            acc = (acc ^ xround(0, v)) * kP1 + kP4;
            acc = (acc ^ xround(0, v2)) * kP1 + kP4;
            acc = (acc ^ xround(0, v3)) * kP1 + kP4;
            acc = (acc ^ xround(0, v4)) * kP1 + kP4;
            acc += (uint64_t)((cb - ca) * 4);
            for (; q + 2 <= cb; q += 2) {
                acc ^= xround(0, lane8(tok, q));
                acc = rotl(acc, 27) * kP1 + kP4;
            }
            if (q < cb) {
                acc ^= (uint64_t)tok(q) * kP1;
                acc = rotl(acc, 23) * kP2 + kP3;
            }
            acc ^= acc >> 33;
            acc *= kP2;
            acc ^= acc >> 29;
            acc *= kP3;
            acc ^= acc >> 32;
            p.fingerprint[s_lk[i]] = acc;
        }
    }
}

// kv_fingerprint: one thread per range [start[k], end[k]).
__global__ void __launch_bounds__(kThreadsCdc) fingerprint_kernel(FingerprintParams p)
{
    const GlobalTokens tok{p.tokens};
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < p.count;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t a = p.start[k], b = p.end[k];
        if (a < 0 || b < a || b > p.total) {
            set_status(p.status, kStatusOutOfRange);
            continue;
        }
        p.fingerprint[k] = xxh64_tokens(tok, a, b, p.seed);
    }
}

} // namespace

int64_t cdc_blocks(int64_t total) { return (total + kTileCdc - 1) / kTileCdc; }

cudaError_t launch_cdc(const CdcParams &p, cudaStream_t stream)
{
    if (p.blocks == 0)
        return cudaSuccess;
    const size_t smem_g = (size_t)kStagePadded * sizeof(uint64_t);
    const size_t smem_t = (size_t)(kTileCdc + kLookback) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(cdc_flags_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_g);
    if (e != cudaSuccess)
        return e;
    cdc_flags_kernel<<<p.blocks, kThreadsCdc, smem_g, stream>>>(p);
    cdc_scan_kernel<<<1, 1024, 0, stream>>>(p);
    cdc_emit_kernel<<<p.blocks, kThreadsCdc, smem_t, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fingerprint(const FingerprintParams &p, cudaStream_t stream)
{
    if (p.count <= 0)
        return cudaSuccess;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    const int64_t want = (p.count + kThreadsCdc - 1) / kThreadsCdc;
    const int grid = (int)max((int64_t)1, min(want, (int64_t)sms * 8));
    fingerprint_kernel<<<grid, kThreadsCdc, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace kvr
