// kv_patch.cu -- relocation with the rank-m patch fused, and the in-place
// patch, for ranks up to 16 (Kamera §2: KV^(B|A) = R(δ)·KV(B|∅) + U_m V_mᵀ).
//
// The patch factors V(l, c) are shared by every token of chunk c in layer l,
// so one block handles one (chunk, layer): each thread owns CPT adjacent
// columns of the row (verbatim part or rotary part) and keeps their V
// factors in registers for the whole chunk.  Rows stream through a ring of
// shared-memory stages filled with cp.async (16 bytes per copy, completion
// by cp.async.wait_group, so no register is held by a load in flight and no
// spin-wait exists); the U rows of each stage are staged the same way.  Per
// row a thread forms Σ_r U(t, r)·V(col, r) for its columns with packed fp32
// FMAs (fma.rn.f32x2), adds it to the copied value or to the unrounded
// rotated value (partner half read from shared memory), rounds once to bf16
// and stores its CPT values to the destination row.
#include "kv_launch.h"
#include "kv_tiles.cuh"

namespace kvr {

// COPY: verbatim columns; NH x D: rotary heads; CPT: columns per thread;
// G: rows per stage; NS: stages in the ring.
template <int COPY_, int NH_, int D_, int CPT_, int G_, int NS_, int MIN_BLOCKS_>
struct PatchGeo {
    static constexpr int COPY = COPY_, NH = NH_, D = D_, CPT = CPT_, G = G_, NS = NS_;
    static constexpr int kMinBlocks = MIN_BLOCKS_;
    static constexpr int ROT = NH * D;
    static constexpr int COLS = COPY + ROT;
    static constexpr int NT = COLS / CPT;               // threads per block
    static constexpr int ROW_BYTES = COLS * 2;
    static constexpr int VEC_PER_ROW = ROW_BYTES / 16;  // 16-byte copies per row
    static constexpr int COPY_VECS = COPY * 2 / 16;
    static constexpr int STAGE_VECS = G * VEC_PER_ROW;
    static constexpr int MMAX = 16;                     // largest rank this kernel takes
    static constexpr int HALF = D / 2;
    static_assert(NT % 32 == 0, "whole warps");
    static_assert(COPY % (32 * CPT) == 0, "warps do not straddle the two parts");
    static_assert(CPT % 2 == 0, "columns come in fp32 pairs");
};

using PatchGeoMla = PatchGeo<512, 1, 64, 2, 8, 4, 2>;   // 288 threads
using PatchGeoGqa = PatchGeo<1024, 8, 128, 4, 4, 4, 1>; // 512 threads

__device__ __forceinline__ void cp_async16(uint32_t smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// acc(2) += u * v(2), one packed fp32x2 FMA.
__device__ __forceinline__ float2 ffma2(float u, float2 v, float2 acc)
{
    unsigned long long a, b, c;
    a = (unsigned long long)__float_as_uint(u) | ((unsigned long long)__float_as_uint(u) << 32);
    b = (unsigned long long)__float_as_uint(v.x) | ((unsigned long long)__float_as_uint(v.y) << 32);
    c = (unsigned long long)__float_as_uint(acc.x) | ((unsigned long long)__float_as_uint(acc.y) << 32);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c) : "l"(a), "l"(b));
    return make_float2(__uint_as_float((uint32_t)c), __uint_as_float((uint32_t)(c >> 32)));
}

template <class P, bool RELOC>
__global__ void __launch_bounds__(P::NT, P::kMinBlocks)
patch_chunk_kernel(const __grid_constant__ RelocParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *ring = smem;                                        // [NS][G][ROW_BYTES]
    float *u_s = reinterpret_cast<float *>(smem + P::NS * P::G * P::ROW_BYTES); // [NS][2][G][MMAX]
    __shared__ int64_t s_src[P::NS + 1][P::G];
    __shared__ int64_t s_dst[P::NS + 1][P::G];

    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const int l = blockIdx.y;
    if (c == 0 && l == 0 && tid == 0) {
        if (p.tok_off[0] != 0 || p.tok_off[p.num_chunks] != p.total_tokens)
            set_status(p.status, kStatusOutOfRange);
    }
    const int64_t t0 = p.tok_off[c];
    const int64_t n = max((int64_t)0, (int64_t)p.tok_off[c + 1] - t0);
    const int32_t req = p.chunk_req[c];
    const bool req_ok = req >= 0 && req < p.num_reqs;
    const int32_t *bt = p.block_tables + (int64_t)(req_ok ? req : 0) * p.max_blocks;
    const int64_t pos0 = p.chunk_dst_pos[c];
    const bool ident = !RELOC || p.delta[c] == 0;
    const int m = p.patch.m;
    const int64_t nstages = (n + P::G - 1) / P::G;

    // this thread's columns
    const int col = tid * P::CPT;
    const int ch = col < P::COPY ? 0 : 1;
    const int cc = ch == 0 ? col : col - P::COPY;
    const bool patched = p.patch.u[ch] != nullptr;
    const int j0 = cc % P::D;
    const bool first = j0 < P::HALF;
    const int partner = ch == 1 ? (first ? cc + P::HALF : cc - P::HALF) : 0;

    // V factors of my columns (registers, whole chunk), as fp32 pairs
    float2 v2[P::CPT / 2][P::MMAX];
#pragma unroll
    for (int e = 0; e < P::CPT / 2; ++e)
#pragma unroll
        for (int r = 0; r < P::MMAX; ++r)
            v2[e][r] = make_float2(0.f, 0.f);
    if (patched) {
        const float *vb = p.patch.v[ch] + (int64_t)l * p.patch.v_ls[ch] +
                          (int64_t)c * p.patch.v_cs[ch];
#pragma unroll
        for (int e = 0; e < P::CPT / 2; ++e) {
            const float *va = vb + (int64_t)(cc + 2 * e) * p.patch.v_cols[ch];
            const float *vbb = va + p.patch.v_cols[ch];
#pragma unroll
            for (int r = 0; r < P::MMAX; r += 4) {
                if (r < m) {
                    const float4 a = __ldg(reinterpret_cast<const float4 *>(va + r));
                    const float4 b = __ldg(reinterpret_cast<const float4 *>(vbb + r));
                    v2[e][r] = make_float2(a.x, b.x);
                    v2[e][r + 1] = make_float2(a.y, b.y);
                    v2[e][r + 2] = make_float2(a.z, b.z);
                    v2[e][r + 3] = make_float2(a.w, b.w);
                }
            }
        }
    }
    // cos/sin of my rotary frequencies (the chunk has one δ)
    float4 cs[P::CPT];
#pragma unroll
    for (int e = 0; e < P::CPT; ++e)
        cs[e] = (ch == 1 && !ident) ? p.table[(int64_t)c * P::HALF + (j0 % P::HALF) + e]
                                    : make_float4(1.f, 0.f, 0.f, 0.f);

    // row metadata of stage s into ring slot s % (NS+1); threads < G
    auto plan = [&](int64_t s) {
        if (tid < P::G) {
            const int64_t i = s * P::G + tid;
            int64_t src = -1, dst = -1;
            if (i < n) {
                if (req_ok)
                    dst = slot_of(bt, p.max_blocks, p.dst.block, p.dst.num_blocks, pos0 + i);
                if (RELOC) {
                    const int64_t sl = p.src_slots[t0 + i];
                    src = (sl >= 0 && sl < p.src.num_slots) ? sl : -1;
                } else {
                    src = dst;
                }
                if (src < 0 || dst < 0) {
                    set_status(p.status, kStatusOutOfRange);
                    src = dst = -1;
                }
            }
            s_src[s % (P::NS + 1)][tid] = src;
            s_dst[s % (P::NS + 1)][tid] = dst;
        }
    };
    const PoolView &sp = RELOC ? p.src : p.dst;
    const char *src_copy = sp.copy + (int64_t)l * sp.copy_ls;
    const char *src_rot = sp.rot + (int64_t)l * sp.rot_ls;
    const uint32_t ring_base = (uint32_t)__cvta_generic_to_shared(ring);
    const uint32_t u_base = (uint32_t)__cvta_generic_to_shared(u_s);
    // issue the copies of stage s (rows and U rows) into buffer s % NS
    auto issue = [&](int64_t s) {
        if (s < nstages) {
            const int slot = (int)(s % (P::NS + 1));
            const int buf = (int)(s % P::NS);
            for (int q = tid; q < P::STAGE_VECS; q += P::NT) {
                const int row = q / P::VEC_PER_ROW, v = q % P::VEC_PER_ROW;
                const int64_t sl = s_src[slot][row];
                if (sl < 0)
                    continue;
                const char *g = v < P::COPY_VECS ? src_copy + sl * sp.copy_ss + v * 16
                                                 : src_rot + sl * sp.rot_ss + (v - P::COPY_VECS) * 16;
                cp_async16(ring_base + (uint32_t)((buf * P::G + row) * P::ROW_BYTES + v * 16), g);
            }
            // U rows: [2][G][m] floats, 4 per copy
            const int uv = m / 4;
            for (int q = tid; q < 2 * P::G * uv; q += P::NT) {
                const int cch = q / (P::G * uv), row = (q / uv) % P::G, r4 = q % uv;
                const int64_t i = s * P::G + row;
                if (p.patch.u[cch] == nullptr || i >= n)
                    continue;
                const float *g = p.patch.u[cch] + (int64_t)l * p.patch.u_ls[cch] +
                                 (t0 + i) * p.patch.u_ts[cch] + r4 * 4;
                cp_async16(u_base + (uint32_t)((((buf * 2 + cch) * P::G + row) * P::MMAX + r4 * 4) * 4), g);
            }
        }
        cp_async_commit();
    };

    for (int s = 0; s < P::NS; ++s)
        plan(s);
    __syncthreads();
    for (int s = 0; s < P::NS - 1; ++s)
        issue(s);

    char *dst_copy = p.dst.copy + (int64_t)l * p.dst.copy_ls;
    char *dst_rot = p.dst.rot + (int64_t)l * p.dst.rot_ls;
    for (int64_t s = 0; s < nstages; ++s) {
        cp_async_wait<P::NS - 2>();
        __syncthreads();
        issue(s + P::NS - 1);
        plan(s + P::NS);
        const int slot = (int)(s % (P::NS + 1));
        const int buf = (int)(s % P::NS);
#pragma unroll 1
        for (int row = 0; row < P::G; ++row) {
            const int64_t d = s_dst[slot][row];
            if (d < 0)
                continue;
            const unsigned char *rb = ring + (buf * P::G + row) * P::ROW_BYTES;
            // patch term of my columns
            float2 acc[P::CPT / 2];
#pragma unroll
            for (int e = 0; e < P::CPT / 2; ++e)
                acc[e] = make_float2(0.f, 0.f);
            if (patched) {
                const float4 *ur =
                    reinterpret_cast<const float4 *>(u_s + ((buf * 2 + ch) * P::G + row) * P::MMAX);
#pragma unroll
                for (int r = 0; r < P::MMAX; r += 4) {
                    if (r < m) {
                        const float4 u = ur[r / 4];
#pragma unroll
                        for (int e = 0; e < P::CPT / 2; ++e) {
                            acc[e] = ffma2(u.x, v2[e][r], acc[e]);
                            acc[e] = ffma2(u.y, v2[e][r + 1], acc[e]);
                            acc[e] = ffma2(u.z, v2[e][r + 2], acc[e]);
                            acc[e] = ffma2(u.w, v2[e][r + 3], acc[e]);
                        }
                    }
                }
            }
            float add[P::CPT];
#pragma unroll
            for (int e = 0; e < P::CPT / 2; ++e) {
                add[2 * e] = acc[e].x;
                add[2 * e + 1] = acc[e].y;
            }
            // my values (and the partner half for a rotation)
            const unsigned char *xp = rb + (ch == 0 ? cc * 2 : P::COPY * 2 + cc * 2);
            uint32_t xw[P::CPT / 2], yw[P::CPT / 2];
#pragma unroll
            for (int e = 0; e < P::CPT / 2; ++e)
                xw[e] = reinterpret_cast<const uint32_t *>(xp)[e];
            uint32_t out[P::CPT / 2];
            if (ch == 1 && !ident) {
                const unsigned char *yp = rb + P::COPY * 2 + partner * 2;
#pragma unroll
                for (int e = 0; e < P::CPT / 2; ++e)
                    yw[e] = reinterpret_cast<const uint32_t *>(yp)[e];
#pragma unroll
                for (int e = 0; e < P::CPT / 2; ++e) {
                    const uint32_t x0 = first ? (xw[e] & 0xFFFFu) : (yw[e] & 0xFFFFu);
                    const uint32_t y0 = first ? (yw[e] & 0xFFFFu) : (xw[e] & 0xFFFFu);
                    const uint32_t x1 = first ? (xw[e] >> 16) : (yw[e] >> 16);
                    const uint32_t y1 = first ? (yw[e] >> 16) : (xw[e] >> 16);
                    out[e] = rotate_one(x0, y0, cs[2 * e], first, add[2 * e]) |
                             (rotate_one(x1, y1, cs[2 * e + 1], first, add[2 * e + 1]) << 16);
                }
            } else if (patched) {
#pragma unroll
                for (int e = 0; e < P::CPT / 2; ++e)
                    out[e] = add_round(xw[e] & 0xFFFFu, add[2 * e]) |
                             (add_round(xw[e] >> 16, add[2 * e + 1]) << 16);
            } else {
#pragma unroll
                for (int e = 0; e < P::CPT / 2; ++e)
                    out[e] = xw[e];
            }
            char *dp = ch == 0 ? dst_copy + d * p.dst.copy_ss + cc * 2
                               : dst_rot + d * p.dst.rot_ss + cc * 2;
            if (P::CPT == 4)
                __stcs(reinterpret_cast<uint2 *>(dp), make_uint2(out[0], out[P::CPT / 2 - 1]));
            else
                __stcs(reinterpret_cast<unsigned int *>(dp), out[0]);
        }
    }
    cp_async_wait<0>();
}

template <class P>
static size_t patch_smem_bytes()
{
    return (size_t)P::NS * P::G * P::ROW_BYTES + (size_t)P::NS * 2 * P::G * P::MMAX * sizeof(float);
}

template <class P, bool RELOC>
static cudaError_t launch_patch_geo(const RelocParams &p, cudaStream_t stream)
{
    const size_t smem = patch_smem_bytes<P>();
    cudaError_t e = cudaFuncSetAttribute(patch_chunk_kernel<P, RELOC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)p.num_chunks, (unsigned)p.src.num_layers);
    patch_chunk_kernel<P, RELOC><<<grid, P::NT, smem, stream>>>(p);
    return cudaGetLastError();
}

bool patch_chunk_supported(const RelocParams &p)
{
    return p.patched && p.patch.m <= 16 && p.src.num_layers <= 65535;
}

cudaError_t launch_patch_chunks(const RelocParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.num_chunks == 0)
        return cudaSuccess;
    if (kind == RowKind::Mla)
        return p.in_place ? launch_patch_geo<PatchGeoMla, false>(p, stream)
                          : launch_patch_geo<PatchGeoMla, true>(p, stream);
    return p.in_place ? launch_patch_geo<PatchGeoGqa, false>(p, stream)
                      : launch_patch_geo<PatchGeoGqa, true>(p, stream);
}

} // namespace kvr
