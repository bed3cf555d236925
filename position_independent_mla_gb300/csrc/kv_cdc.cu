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
// Kernels (one call):
//   1. cdc_flags_kernel: a block owns 8192 positions; it stages G for them
//      and the 63 before them in shared memory (coalesced), each thread rolls
//      the hash over its 32 positions (after 63 warm-up steps that rebuild
//      the window) and keeps one bit per position; per-block counts.
//   2. cdc_scan_kernel: one block turns the counts into offsets and the total.
//   3. cdc_emit_kernel: every set bit becomes a chunk end, in stream order.
//   4. fingerprint_kernel: one thread per chunk hashes its tokens.
#include "kv_device.cuh"
#include "kv_launch.h"

namespace kvr {
namespace {

constexpr int kThreadsCdc = 256;
constexpr int kRun = 32;                         // positions per thread
constexpr int kTileCdc = kThreadsCdc * kRun;     // positions per block
constexpr int kWindow = 64;                      // tokens a Gear hash holds
constexpr int kHalo = kWindow - 1;
constexpr int kStageEntries = kTileCdc + kHalo;
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

// Stream holding position q: the largest s with stream_off[s] <= q (empty
// streams share their offset with the next one, so this is the non-empty one).
__device__ __forceinline__ int stream_of(const int64_t *off, int num_streams, int64_t q)
{
    int lo = 0, hi = num_streams - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= q)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kThreadsCdc) cdc_flags_kernel(const __grid_constant__ CdcParams p)
{
    extern __shared__ uint64_t s_g[];
    __shared__ int64_t s_warp[kThreadsCdc / 32];
    const int tid = threadIdx.x;
    const int64_t tile0 = (int64_t)blockIdx.x * kTileCdc;
    const int64_t lo = tile0 - kHalo;
    const int64_t hi = min(tile0 + kTileCdc, p.total);

    if (blockIdx.x == 0 && tid == 0) {
        if (p.stream_off[0] != 0 || p.stream_off[p.num_streams] != p.total)
            set_status(p.status, kStatusOutOfRange);
    }
    for (int64_t q = max(lo, (int64_t)0) + tid; q < hi; q += kThreadsCdc)
        s_g[staged((int)(q - lo))] = gear_value(p.gear_seed, (uint32_t)p.tokens[q]);
    __syncthreads();

    const int64_t p0 = tile0 + (int64_t)tid * kRun;
    uint32_t flags = 0;
    if (p0 < p.total) {
        int s = stream_of(p.stream_off, p.num_streams, p0);
        int64_t s_start = p.stream_off[s], s_end = p.stream_off[s + 1];
        uint64_t h = 0;
        // rebuild the window: the (up to 63) tokens of this stream before p0
        for (int64_t q = max(s_start, p0 - kHalo); q < p0; ++q)
            h = 2u * h + s_g[staged((int)(q - lo))];
        const int64_t pend = min(p0 + kRun, p.total);
        for (int64_t q = p0; q < pend; ++q) {
            while (q >= s_end && s + 1 < p.num_streams) { // the next non-empty stream
                ++s;
                s_start = p.stream_off[s];
                s_end = p.stream_off[s + 1];
                h = 0;
            }
            h = 2u * h + s_g[staged((int)(q - lo))];
            if (h < p.threshold || q == s_end - 1)
                flags |= 1u << (int)(q - p0);
        }
    }
    p.flags[(int64_t)blockIdx.x * kThreadsCdc + tid] = flags;

    int64_t c = __popc(flags);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if ((tid & 31) == 0)
        s_warp[tid >> 5] = c;
    __syncthreads();
    if (tid == 0) {
        int64_t t = 0;
#pragma unroll
        for (int w = 0; w < kThreadsCdc / 32; ++w)
            t += s_warp[w];
        p.block_count[blockIdx.x] = t;
    }
}

// Exclusive scan of the per-block counts (one block of 1024 threads).
__global__ void __launch_bounds__(1024) cdc_scan_kernel(const __grid_constant__ CdcParams p)
{
    __shared__ int64_t s_part[1024];
    const int tid = threadIdx.x;
    const int per = (p.blocks + 1023) / 1024;
    const int b0 = min(tid * per, p.blocks), b1 = min(b0 + per, p.blocks);
    int64_t sum = 0;
    for (int b = b0; b < b1; ++b)
        sum += p.block_count[b];
    s_part[tid] = sum;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) { // inclusive Hillis-Steele scan
        const int64_t v = tid >= o ? s_part[tid - o] : 0;
        __syncthreads();
        s_part[tid] += v;
        __syncthreads();
    }
    int64_t run = s_part[tid] - sum;
    for (int b = b0; b < b1; ++b) {
        p.block_off[b] = run;
        run += p.block_count[b];
    }
    if (tid == 1023) {
        *p.num_chunks = s_part[1023];
        if (s_part[1023] > p.max_chunks)
            set_status(p.status, kStatusCapacity);
    }
}

// Every set flag bit becomes a chunk end (exclusive, a global token offset).
__global__ void __launch_bounds__(kThreadsCdc) cdc_emit_kernel(const __grid_constant__ CdcParams p)
{
    __shared__ int64_t s_warp[kThreadsCdc / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t flags = p.flags[(int64_t)blockIdx.x * kThreadsCdc + tid];
    const int c = __popc(flags);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        s_warp[warp] = incl;
    __syncthreads();
    int64_t base = p.block_off[blockIdx.x];
    for (int w = 0; w < warp; ++w)
        base += s_warp[w];
    int64_t k = base + incl - c;
    const int64_t p0 = (int64_t)blockIdx.x * kTileCdc + (int64_t)tid * kRun;
    uint32_t f = flags;
    while (f) {
        const int j = __ffs(f) - 1;
        f &= f - 1;
        if (k < p.max_chunks)
            p.chunk_end[k] = p0 + j + 1;
        ++k;
    }
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

// Eight bytes = tokens t[0], t[1] as little-endian words.
__device__ __forceinline__ uint64_t lane8(const int32_t *t)
{
    return (uint64_t)(uint32_t)__ldg(t) | ((uint64_t)(uint32_t)__ldg(t + 1) << 32);
}

__device__ uint64_t xxh64_tokens(const int32_t *t, int64_t n, uint64_t seed)
{
    const int64_t len = n * 4;
    int64_t i = 0; // next token
    uint64_t acc;
    if (len >= 32) {
        uint64_t v1 = seed + kP1 + kP2, v2 = seed + kP2, v3 = seed, v4 = seed - kP1;
        for (; i + 8 <= n; i += 8) {
            v1 = xround(v1, lane8(t + i));
            v2 = xround(v2, lane8(t + i + 2));
            v3 = xround(v3, lane8(t + i + 4));
            v4 = xround(v4, lane8(t + i + 6));
        }
        acc = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
        acc = (acc ^ xround(0, v1)) * kP1 + kP4;
        acc = (acc ^ xround(0, v2)) * kP1 + kP4;
        acc = (acc ^ xround(0, v3)) * kP1 + kP4;
        acc = (acc ^ xround(0, v4)) * kP1 + kP4;
    } else {
        acc = seed + kP5;
    }
    acc += (uint64_t)len;
    for (; i + 2 <= n; i += 2) {
        acc ^= xround(0, lane8(t + i));
        acc = rotl(acc, 27) * kP1 + kP4;
    }
    if (i < n) { // one 4-byte word left (token counts leave no single bytes)
        acc ^= (uint64_t)(uint32_t)__ldg(t + i) * kP1;
        acc = rotl(acc, 23) * kP2 + kP3;
    }
    acc ^= acc >> 33;
    acc *= kP2;
    acc ^= acc >> 29;
    acc *= kP3;
    acc ^= acc >> 32;
    return acc;
}

// One thread per range; ranges [start[k], end[k]), or, with start == NULL,
// consecutive chunks (start = the previous end, 0 for the first).  With
// `count` the number of ranges is min(*count, cap), read on the device.
__global__ void __launch_bounds__(kThreadsCdc) fingerprint_kernel(FingerprintParams p)
{
    const int64_t n = p.count ? min(*p.count, p.cap) : p.cap;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t a = p.start ? p.start[k] : (k ? p.end[k - 1] : 0);
        const int64_t b = p.end[k];
        if (a < 0 || b < a || b > p.total) {
            set_status(p.status, kStatusOutOfRange);
            continue;
        }
        p.fingerprint[k] = xxh64_tokens(p.tokens + a, b - a, p.seed);
    }
}

cudaError_t launch_fp(const FingerprintParams &p, cudaStream_t stream)
{
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    const int64_t want = (p.cap + kThreadsCdc - 1) / kThreadsCdc;
    const int grid = (int)max((int64_t)1, min(want, (int64_t)sms * 8));
    fingerprint_kernel<<<grid, kThreadsCdc, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace

int64_t cdc_blocks(int64_t total) { return (total + kTileCdc - 1) / kTileCdc; }

cudaError_t launch_cdc(const CdcParams &p, cudaStream_t stream)
{
    if (p.blocks == 0)
        return cudaSuccess;
    const size_t smem = (size_t)kStagePadded * sizeof(uint64_t);
    cudaError_t e = cudaFuncSetAttribute(cdc_flags_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cdc_flags_kernel<<<p.blocks, kThreadsCdc, smem, stream>>>(p);
    cdc_scan_kernel<<<1, 1024, 0, stream>>>(p);
    cdc_emit_kernel<<<p.blocks, kThreadsCdc, 0, stream>>>(p);
    FingerprintParams f{};
    f.tokens = p.tokens;
    f.total = p.total;
    f.start = nullptr;
    f.end = p.chunk_end;
    f.count = p.num_chunks;
    f.cap = min(p.max_chunks, p.total);
    f.seed = p.fp_seed;
    f.fingerprint = p.fingerprint;
    f.status = p.status;
    if (f.cap > 0) {
        e = launch_fp(f, stream);
        if (e != cudaSuccess)
            return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_fingerprint(const FingerprintParams &p, cudaStream_t stream)
{
    return p.cap > 0 ? launch_fp(p, stream) : cudaSuccess;
}

} // namespace kvr
