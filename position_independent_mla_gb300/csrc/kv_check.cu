// kv_check.cu -- debug checks of the caller contracts the in-place kernels
// rely on (kv_set_debug_checks): a relocation inside one pool must not write
// a slot that the same call reads, and a splice's block-table entries must
// name distinct blocks.  Each check marks a bitmap in the caller's workspace
// and sets KV_ERR_OVERLAP in the status word; the call's row-moving kernels
// read that word first and then store nothing.
#include <algorithm>

#include "kv_device.cuh"
#include "kv_launch.h"

namespace kvr {

namespace {

constexpr int kCheckThreads = 256;
constexpr int64_t kCheckMaxBlocks = 152 * 8; // grid-stride beyond one wave

__device__ __forceinline__ bool test_and_mark(uint32_t *bitmap, int64_t i)
{
    const uint32_t bit = 1u << (i & 31);
    return (atomicOr(bitmap + (i >> 5), bit) & bit) != 0u;
}

__device__ __forceinline__ bool is_marked(const uint32_t *bitmap, int64_t i)
{
    return (bitmap[i >> 5] >> (i & 31)) & 1u;
}

// Every source slot inside the destination pool's range.
__global__ void overlap_mark_kernel(const __grid_constant__ OverlapParams p)
{
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < p.total_tokens;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t s = p.src_slots[t];
        if (s >= 0 && s < p.num_slots)
            test_and_mark(p.bitmap, s);
    }
}

// Every destination slot against the marked source slots.  Indices that are
// out of range are left to the relocation kernel, which reports them.
__global__ void overlap_test_kernel(const __grid_constant__ OverlapParams p)
{
    bool hit = false;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < p.total_tokens;
         t += (int64_t)gridDim.x * blockDim.x) {
        int lo = 0, hi = p.num_chunks - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tok_off[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int64_t off = t - p.tok_off[lo];
        const int32_t req = p.chunk_req[lo];
        if (off < 0 || t >= p.tok_off[lo + 1] || req < 0 || req >= p.num_reqs)
            continue;
        const int64_t dst = slot_of(p.block_tables + (int64_t)req * p.max_blocks, p.max_blocks,
                                    p.block, p.num_blocks, (int64_t)p.chunk_dst_pos[lo] + off);
        if (dst >= 0 && is_marked(p.bitmap, dst))
            hit = true;
    }
    if (hit)
        set_status(p.status, kStatusOverlap);
}

// Every used block-table entry marked once; a second mark is a duplicate.
__global__ void dup_block_kernel(const __grid_constant__ DupBlockParams p)
{
    const int64_t n = (int64_t)p.rows * p.max_blocks;
    bool dup = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / p.max_blocks, j = i % p.max_blocks;
        if (j >= p.used[row])
            continue;
        const int64_t blk = p.block_tables[i];
        if (blk >= 0 && blk < p.num_blocks && test_and_mark(p.bitmap, blk))
            dup = true;
    }
    if (dup)
        set_status(p.status, kStatusOverlap);
}

unsigned grid_for(int64_t n)
{
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + kCheckThreads - 1) / kCheckThreads,
                                                            kCheckMaxBlocks));
}

} // namespace

cudaError_t launch_overlap_check(const OverlapParams &p, cudaStream_t stream)
{
    if (p.total_tokens <= 0)
        return cudaSuccess;
    const unsigned g = grid_for(p.total_tokens);
    overlap_mark_kernel<<<g, kCheckThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    overlap_test_kernel<<<g, kCheckThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_dup_block_check(const DupBlockParams &p, cudaStream_t stream)
{
    const int64_t n = (int64_t)p.rows * p.max_blocks;
    if (n <= 0)
        return cudaSuccess;
    dup_block_kernel<<<grid_for(n), kCheckThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace kvr
