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
// G: rows per stage; NS: stages in the ring.  SPLIT: one block per channel
// (verbatim part or rotary part, which must then have the same width)
// instead of one block covering the whole row.
template <int COPY_, int NH_, int D_, int CPT_, int G_, int NS_, int MIN_BLOCKS_, bool SPLIT_>
struct PatchGeo {
    static constexpr int COPY = COPY_, NH = NH_, D = D_, CPT = CPT_, G = G_, NS = NS_;
    static constexpr int kMinBlocks = MIN_BLOCKS_;
    static constexpr bool SPLIT = SPLIT_;
    static constexpr int ROT = NH * D;
    static constexpr int COLS = SPLIT ? COPY : COPY + ROT; // columns a block covers
    static constexpr int NT = COLS / CPT;                 // threads per block
    static constexpr int ROW_BYTES = COLS * 2;            // bytes of a row a block stages
    static constexpr int VEC_PER_ROW = ROW_BYTES / 16;    // 16-byte copies per row
    static constexpr int COPY_VECS = SPLIT ? VEC_PER_ROW : COPY * 2 / 16;
    static constexpr int STAGE_VECS = G * VEC_PER_ROW;
    static constexpr int NCH = SPLIT ? 1 : 2;             // channels a block stages U for
    static constexpr int MMAX = 16;                       // largest rank this kernel takes
    static constexpr int HALF = D / 2;
    static_assert(NT % 32 == 0, "whole warps");
    static_assert(SPLIT ? COPY == ROT : COPY % (32 * CPT) == 0, "channel layout");
    static_assert(CPT % 2 == 0, "columns come in fp32 pairs");
    static_assert(G % 2 == 0, "rows are processed in pairs");
};

using PatchGeoMla = PatchGeo<512, 1, 64, 2, 8, 4, 2, false>;  // 288 threads, c_KV + k_pe
using PatchGeoGqa = PatchGeo<1024, 8, 128, 4, 8, 4, 2, true>; // 256 threads per channel

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

// Two fp32 values in one 64-bit register pair (the operand form of the
// packed fp32x2 instructions).
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float a, float b)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float2 unpack2(f32x2 r)
{
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
    return make_float2(a, b);
}

// acc += uu * v on both halves: one fma.rn.f32x2.
__device__ __forceinline__ void ffma2(f32x2 &acc, f32x2 uu, f32x2 v)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(uu), "l"(v));
}

template <class P, bool RELOC>
__global__ void __launch_bounds__(P::NT, P::kMinBlocks)
patch_chunk_kernel(const __grid_constant__ RelocParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *ring = smem; // [NS][G][ROW_BYTES]
    float *u_s = reinterpret_cast<float *>(smem + P::NS * P::G * P::ROW_BYTES); // [NS][NCH][G][MMAX]
    __shared__ int64_t s_src[P::NS + 1][P::G];
    __shared__ int64_t s_dst[P::NS + 1][P::G];

    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const int l = blockIdx.y;
    if (c == 0 && l == 0 && blockIdx.z == 0 && tid == 0) {
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

    // this thread's channel and columns
    const int col = tid * P::CPT;
    const int ch = P::SPLIT ? (int)blockIdx.z : (col < P::COPY ? 0 : 1);
    const int cc = (P::SPLIT || ch == 0) ? col : col - P::COPY;
    const int ch0 = P::SPLIT ? ch : 0;           // first channel staged by this block
    const bool patched = p.patch.u[ch] != nullptr;
    const int j0 = cc % P::D;
    const bool first = j0 < P::HALF;
    const int partner = ch == 1 ? (first ? cc + P::HALF : cc - P::HALF) : 0;
    // byte offset of channel ch inside a staged row
    const int ch_off = (P::SPLIT || ch == 0) ? 0 : P::COPY * 2;

    // V factors of my columns (registers, whole chunk), as rank pairs:
    // v2[e][q] = (V(col_e, 2q), V(col_e, 2q+1))
    f32x2 v2[P::CPT][P::MMAX / 2];
#pragma unroll
    for (int e = 0; e < P::CPT; ++e)
#pragma unroll
        for (int q = 0; q < P::MMAX / 2; ++q)
            v2[e][q] = 0ull;
    if (patched) {
        const float *vb = p.patch.v[ch] + (int64_t)l * p.patch.v_ls[ch] +
                          (int64_t)c * p.patch.v_cs[ch];
#pragma unroll
        for (int e = 0; e < P::CPT; ++e) {
            const float *va = vb + (int64_t)(cc + e) * p.patch.v_cols[ch];
#pragma unroll
            for (int r = 0; r < P::MMAX; r += 4) {
                if (r < m) {
                    const float4 a = __ldg(reinterpret_cast<const float4 *>(va + r));
                    v2[e][r / 2] = pack2(a.x, a.y);
                    v2[e][r / 2 + 1] = pack2(a.z, a.w);
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
                const bool in_copy = P::SPLIT ? ch == 0 : v < P::COPY_VECS;
                const int vo = P::SPLIT ? v : (in_copy ? v : v - P::COPY_VECS);
                const char *g = in_copy ? src_copy + sl * sp.copy_ss + vo * 16
                                        : src_rot + sl * sp.rot_ss + vo * 16;
                cp_async16(ring_base + (uint32_t)((buf * P::G + row) * P::ROW_BYTES + v * 16), g);
            }
            // U rows: [NCH][G][m] floats, 4 per copy
            const int uv = m / 4;
            for (int q = tid; q < P::NCH * P::G * uv; q += P::NT) {
                const int k = q / (P::G * uv), row = (q / uv) % P::G, r4 = q % uv;
                const int cch = ch0 + k;
                const int64_t i = s * P::G + row;
                if (p.patch.u[cch] == nullptr || i >= n)
                    continue;
                const float *g = p.patch.u[cch] + (int64_t)l * p.patch.u_ls[cch] +
                                 (t0 + i) * p.patch.u_ts[cch] + r4 * 4;
                cp_async16(u_base + (uint32_t)((((buf * P::NCH + k) * P::G + row) * P::MMAX + r4 * 4) * 4), g);
            }
        }
        cp_async_commit();
    };

    for (int s = 0; s < P::NS; ++s)
        plan(s);
    __syncthreads();
    for (int s = 0; s < P::NS - 1; ++s)
        issue(s);

    char *dst_base = ch == 0 ? p.dst.copy + (int64_t)l * p.dst.copy_ls
                             : p.dst.rot + (int64_t)l * p.dst.rot_ls;
    const int64_t dst_ss = ch == 0 ? p.dst.copy_ss : p.dst.rot_ss;
    for (int64_t s = 0; s < nstages; ++s) {
        cp_async_wait<P::NS - 2>();
        __syncthreads();
        issue(s + P::NS - 1);
        plan(s + P::NS);
        const int slot = (int)(s % (P::NS + 1));
        const int buf = (int)(s % P::NS);
        // two rows per step: independent FMA and rounding chains interleave
#pragma unroll 1
        for (int row0 = 0; row0 < P::G; row0 += 2) {
            int64_t d[2];
            float add[2][P::CPT];
            const unsigned char *rb[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                d[k] = s_dst[slot][row0 + k];
                rb[k] = ring + (buf * P::G + row0 + k) * P::ROW_BYTES;
            }
            if (patched) {
                f32x2 acc[2][P::CPT];
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int e = 0; e < P::CPT; ++e)
                        acc[k][e] = 0ull;
                const f32x2 *ur0 = reinterpret_cast<const f32x2 *>(
                    u_s + ((buf * P::NCH + (ch - ch0)) * P::G + row0) * P::MMAX);
                const f32x2 *ur1 = ur0 + P::MMAX / 2;
#pragma unroll
                for (int q = 0; q < P::MMAX / 2; ++q) {
                    if (2 * q < m) {
                        const f32x2 u0 = ur0[q], u1 = ur1[q];
#pragma unroll
                        for (int e = 0; e < P::CPT; ++e) {
                            ffma2(acc[0][e], u0, v2[e][q]);
                            ffma2(acc[1][e], u1, v2[e][q]);
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int e = 0; e < P::CPT; ++e) {
                        const float2 a = unpack2(acc[k][e]);
                        add[k][e] = a.x + a.y;
                    }
            } else {
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int e = 0; e < P::CPT; ++e)
                        add[k][e] = 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (d[k] < 0)
                    continue;
                // my values (and the partner half for a rotation)
                const unsigned char *xp = rb[k] + ch_off + cc * 2;
                uint32_t xw[P::CPT / 2], yw[P::CPT / 2], out[P::CPT / 2];
#pragma unroll
                for (int e = 0; e < P::CPT / 2; ++e)
                    xw[e] = reinterpret_cast<const uint32_t *>(xp)[e];
                if (ch == 1 && !ident) {
                    const unsigned char *yp = rb[k] + ch_off + partner * 2;
#pragma unroll
                    for (int e = 0; e < P::CPT / 2; ++e)
                        yw[e] = reinterpret_cast<const uint32_t *>(yp)[e];
#pragma unroll
                    for (int e = 0; e < P::CPT / 2; ++e) {
                        const uint32_t x0 = first ? (xw[e] & 0xFFFFu) : (yw[e] & 0xFFFFu);
                        const uint32_t y0 = first ? (yw[e] & 0xFFFFu) : (xw[e] & 0xFFFFu);
                        const uint32_t x1 = first ? (xw[e] >> 16) : (yw[e] >> 16);
                        const uint32_t y1 = first ? (yw[e] >> 16) : (xw[e] >> 16);
                        if (patched)
                            out[e] = rotate_add_fast(x0, y0, cs[2 * e], first, add[k][2 * e]) |
                                     (rotate_add_fast(x1, y1, cs[2 * e + 1], first,
                                                      add[k][2 * e + 1]) << 16);
                        else
                            out[e] = rotate_one(x0, y0, cs[2 * e], first, 0.0f) |
                                     (rotate_one(x1, y1, cs[2 * e + 1], first, 0.0f) << 16);
                    }
                } else if (patched) {
#pragma unroll
                    for (int e = 0; e < P::CPT / 2; ++e)
                        out[e] = bf16_rne(bf16_lo(xw[e]) + add[k][2 * e]) |
                                 (bf16_rne(bf16_hi(xw[e]) + add[k][2 * e + 1]) << 16);
                } else {
#pragma unroll
                    for (int e = 0; e < P::CPT / 2; ++e)
                        out[e] = xw[e];
                }
                char *dp = dst_base + d[k] * dst_ss + cc * 2;
                if (P::CPT == 4)
                    __stcs(reinterpret_cast<uint2 *>(dp), make_uint2(out[0], out[P::CPT / 2 - 1]));
                else
                    __stcs(reinterpret_cast<unsigned int *>(dp), out[0]);
            }
        }
    }
    cp_async_wait<0>();
}

template <class P>
static size_t patch_smem_bytes()
{
    return (size_t)P::NS * P::G * P::ROW_BYTES +
           (size_t)P::NS * P::NCH * P::G * P::MMAX * sizeof(float);
}

template <class P, bool RELOC>
static cudaError_t launch_patch_geo(const RelocParams &p, cudaStream_t stream)
{
    const size_t smem = patch_smem_bytes<P>();
    cudaError_t e = cudaFuncSetAttribute(patch_chunk_kernel<P, RELOC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)p.num_chunks, (unsigned)p.src.num_layers, P::SPLIT ? 2u : 1u);
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
