// kv_tiles.cuh -- moving a tile of KV rows through registers.
//
// A tile is T rows of one layer.  Each row is CV 16-byte vectors of the
// verbatim part followed (in another array, possibly) by NH rotary heads of
// 2*HV 16-byte vectors.  Work items are single 16-byte vectors, spread over
// the kThreads threads of the block so that one warp instruction touches
// 512 contiguous-per-row bytes.  Rotary items are numbered so that the two
// halves of a head sit in lanes l and l ^ HV of the same warp: a lane loads
// its own half and receives the partner half with a warp shuffle, so every
// byte of the row is loaded exactly once.
#pragma once

#include "kv_device.cuh"
#include "kv_launch.h"

namespace kvr {

template <int T_, int CV_, int NH_, int HV_, int MIN_BLOCKS_>
struct Geo {
    static constexpr int T = T_;
    static constexpr int kMinBlocks = MIN_BLOCKS_; // resident blocks per SM to aim for
    static constexpr int CV = CV_;          // verbatim vectors per row
    static constexpr int NH = NH_;          // rotary heads
    static constexpr int HV = HV_;          // vectors per half head
    static constexpr int kHalf = HV * 8;    // frequencies per head
    static constexpr int kRotW = NH * 2 * HV; // rotary vectors per row
    static constexpr int kCopyItems = T * CV;
    static constexpr int kRotItems = T * kRotW;
    static constexpr int kCopyPer = (kCopyItems + kThreads - 1) / kThreads;
    static constexpr int kRotPer = (kRotItems + kThreads - 1) / kThreads;
    // cos/sin rows in shared memory are stored transposed -- entry e of the
    // 8 frequencies of vector group vv at e*HV + vv -- and padded by 4
    // entries, so the lanes of a warp read them without bank conflicts.
    static constexpr int kCsRow = kHalf + 4;
    static __device__ __forceinline__ int cs_index(int f) { return (f % 8) * HV + f / 8; }
    // Pair-packed order (rotate_vec_packed): frequency f = 8vv + e feeds
    // component (e & 1) of the c1/s1 entry (e & ~1)*HV + vv and of the c2/s2
    // entry (e | 1)*HV + vv -- the same HV*8 entries, regrouped by word.
    static __device__ __forceinline__ void stage_packed(float4 *row, int f, float4 q)
    {
        const int vv = f / 8, e = f % 8, o = e & 1;
        float *a = reinterpret_cast<float *>(row + (e & ~1) * HV + vv);
        float *b = reinterpret_cast<float *>(row + (e | 1) * HV + vv);
        a[o] = q.x;     // c1
        a[2 + o] = q.z; // s1
        b[o] = q.y;     // c2
        b[2 + o] = q.w; // s2
    }
    static_assert(32 % (2 * HV) == 0, "a rotary head's vectors must tile a warp");
    static_assert(kThreads % (2 * HV) == 0, "partner lanes must stay in one item round");
};

// MLA rows: c_KV 512 + k_pe 64 (DeepSeek-V2/V3 shape).
using GeoMla = Geo<kTileMla, 64, 1, 4, 4>;
// GQA rows: V 8x128 + K 8x128 (Llama-3-8B shape).
using GeoGqa = Geo<kTileGqa, 128, 8, 8, 2>;
// GQA rows with 4 KV heads: V 4x128 + K 4x128 (Qwen2.5-7B shape).
using GeoGqa4 = Geo<kTileGqa4, 64, 4, 8, 2>;
// MHA rows: V 32x128 + K 32x128 (Llama-2-7B shape).
using GeoMha = Geo<kTileMha, 512, 32, 8, 2>;

// The in-place passes (the ticketed splice, the block-table remap) are
// limited by latency -- the rotation's dependent arithmetic, the splice's
// waits -- rather than by bytes in flight: multi-head rows take tiles of
// half the rows there, four rotary vectors per thread and four blocks
// (32 warps) per SM.
using GeoGqaInPlace = Geo<kInPlaceTileGqa, 128, 8, 8, 4>;
using GeoGqa4InPlace = Geo<kInPlaceTileGqa4, 64, 4, 8, 4>;
using GeoMhaInPlace = Geo<kInPlaceTileMha, 512, 32, 8, 4>;

// Multi-head rows (GQA, MHA: rotation is half of every row) without a
// patch term, in rotate-half pairing, take the pair-packed rotation; the
// others (MLA's single 64-wide head, patched or interleaved rows) keep one
// (c1, c2, s1, s2) entry per frequency -- except in passes that move only
// the rotary part (ROT_ONLY), where the rotation is all the work and MLA
// rows take the pair-packed rotation too.
template <class G, bool PATCH, bool IL, bool ROT_ONLY = false>
struct CsOrder {
    static constexpr bool kPacked = !PATCH && !IL && (G::NH > 1 || ROT_ONLY);
};

// Write table entry q of frequency f into a shared-memory cos/sin row.
template <class G, bool PACKED>
__device__ __forceinline__ void stage_cs(float4 *row, int f, float4 q)
{
    if (PACKED)
        G::stage_packed(row, f, q);
    else
        row[G::cs_index(f)] = q;
}

template <class G>
struct GeoTag {
    using type = G;
};

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// Call f(BoolTag<b>{}) with b as a compile-time constant.
template <class F>
cudaError_t with_bool(bool b, F &&f)
{
    return b ? f(BoolTag<true>{}) : f(BoolTag<false>{});
}

// Call f(GeoTag<G>{}) with the tile geometry of `kind`.
template <class F>
cudaError_t with_geo(RowKind kind, F &&f)
{
    switch (kind) {
    case RowKind::Mla:
        return f(GeoTag<GeoMla>{});
    case RowKind::Gqa:
        return f(GeoTag<GeoGqa>{});
    case RowKind::Gqa4:
        return f(GeoTag<GeoGqa4>{});
    case RowKind::Mha:
        return f(GeoTag<GeoMha>{});
    }
    return cudaErrorInvalidValue;
}

// with_geo for the in-place passes (tile rows as inplace_tile_rows).
template <class F>
cudaError_t with_inplace_geo(RowKind kind, F &&f)
{
    switch (kind) {
    case RowKind::Mla:
        return f(GeoTag<GeoMla>{});
    case RowKind::Gqa:
        return f(GeoTag<GeoGqaInPlace>{});
    case RowKind::Gqa4:
        return f(GeoTag<GeoGqa4InPlace>{});
    case RowKind::Mha:
        return f(GeoTag<GeoMhaInPlace>{});
    }
    return cudaErrorInvalidValue;
}

// Where the rows of a tile live for one layer: row r's verbatim part starts
// at cbase + idx[r]*cstride, its rotary part at rbase + idx[r]*rstride
// (bytes); idx[r] < 0 marks a row that is skipped.
struct RowsAt {
    const char *cbase;
    int64_t cstride;
    const char *rbase;
    int64_t rstride;
};

template <class G>
struct TileRegs {
    uint4 c[G::kCopyPer];
    uint4 r[G::kRotPer];
};

// COPY = false leaves the verbatim part alone (rotary part only).
template <class G, bool COPY = true>
__device__ __forceinline__ void load_tile(const RowsAt &at, const int64_t *idx, TileRegs<G> &regs)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int k = 0; k < G::kCopyPer; ++k) {
        const int i = tid + k * kThreads;
        regs.c[k] = make_uint4(0u, 0u, 0u, 0u);
        if (COPY && i < G::kCopyItems) {
            const int row = i / G::CV, v = i % G::CV;
            const int64_t s = idx[row];
            if (s >= 0)
                regs.c[k] = ld_stream(at.cbase + s * at.cstride + v * 16);
        }
    }
#pragma unroll
    for (int k = 0; k < G::kRotPer; ++k) {
        const int i = tid + k * kThreads;
        regs.r[k] = make_uint4(0u, 0u, 0u, 0u);
        if (i < G::kRotItems) {
            const int row = i / G::kRotW, w = i % G::kRotW;
            const int64_t s = idx[row];
            if (s >= 0)
                regs.r[k] = ld_stream(at.rbase + s * at.rstride + w * 16);
        }
    }
}

// A data dependency on every loaded word: the block barrier that follows
// is then reached only after all loads of the tile have returned.
template <class G>
__device__ __forceinline__ uint32_t fold_tile(const TileRegs<G> &regs)
{
    uint32_t f = 0;
#pragma unroll
    for (int k = 0; k < G::kCopyPer; ++k)
        f ^= regs.c[k].x ^ regs.c[k].y ^ regs.c[k].z ^ regs.c[k].w;
#pragma unroll
    for (int k = 0; k < G::kRotPer; ++k)
        f ^= regs.r[k].x ^ regs.r[k].y ^ regs.r[k].z ^ regs.r[k].w;
    return f;
}

// Patch context of a tile (relocation only).
struct PatchAt {
    const PatchView *pv;
    int layer;
    const int64_t *tok;   // per row: token index in the call
    const int32_t *chunk; // per row: chunk index
};

// Σ_r U(l, t, r)·V(l, c, col0 + e, r) for e < 8, r ascending, fp32.
__device__ __forceinline__ void patch_terms(const PatchView &pv, int ch, int l, int64_t t,
                                            int32_t c, int col0, float add[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e)
        add[e] = 0.0f;
    if (pv.u[ch] == nullptr)
        return;
    const float *u = pv.u[ch] + (int64_t)l * pv.u_ls[ch] + t * pv.u_ts[ch];
    const float *v = pv.v[ch] + (int64_t)l * pv.v_ls[ch] + (int64_t)c * pv.v_cs[ch] +
                     (int64_t)col0 * pv.v_cols[ch];
    for (int r = 0; r < pv.m; r += 4) {
        const float4 uu = __ldg(reinterpret_cast<const float4 *>(u + r));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 vv = __ldg(reinterpret_cast<const float4 *>(v + e * pv.v_cols[ch] + r));
            float a = add[e];
            a = fmaf(uu.x, vv.x, a);
            a = fmaf(uu.y, vv.y, a);
            a = fmaf(uu.z, vv.z, a);
            a = fmaf(uu.w, vv.w, a);
            add[e] = a;
        }
    }
}

// Interleaved pairing: the 16-byte vector v of a head holds pairs
// (x[8v+2i], x[8v+2i+1]) of frequencies 4v+i, i < 4, one pair per 32-bit
// word, so no partner lane is needed.  cs_row is the row's transposed
// cos/sin table (entry of frequency f at Geo::cs_index(f)).
template <class G>
__device__ __forceinline__ uint4 rotate_vec_il(uint4 x, const float4 *cs_row, int v,
                                               const float *add)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 q = cs_row[G::cs_index(4 * v + i)];
        const uint32_t even = w[i] & 0xFFFFu, odd = w[i] >> 16;
        out[i] = rotate_one(even, odd, q, true, add[2 * i]) |
                 (rotate_one(even, odd, q, false, add[2 * i + 1]) << 16);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Write a loaded tile: verbatim vectors as they are (plus the patch),
// rotary vectors turned by the row's cos/sin (a transposed table row at
// cs + row*cs_row_stride, see Geo::cs_index) unless the row is marked
// identity.
// IL: the rotary pairs are interleaved (x[2j], x[2j+1]) instead of rotate-half.
template <class G, bool PATCH, bool COPY = true, bool IL = false,
          bool PACKED = CsOrder<G, PATCH, IL>::kPacked>
__device__ __forceinline__ void store_tile(const RowsAt &at, const int64_t *idx,
                                           const TileRegs<G> &regs, const float4 *cs,
                                           int cs_row_stride, const int32_t *ident,
                                           const PatchAt &pa)
{
    const int tid = threadIdx.x;
    float add[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        add[e] = 0.0f;
#pragma unroll
    for (int k = 0; k < G::kCopyPer; ++k) {
        const int i = tid + k * kThreads;
        if (COPY && i < G::kCopyItems) {
            const int row = i / G::CV, v = i % G::CV;
            const int64_t s = idx[row];
            if (s >= 0) {
                uint4 out = regs.c[k];
                if (PATCH) {
                    patch_terms(*pa.pv, 0, pa.layer, pa.tok[row], pa.chunk[row], v * 8, add);
                    if (pa.pv->u[0] != nullptr)
                        out = add_vec(out, add);
                }
                st_stream(const_cast<char *>(at.cbase) + s * at.cstride + v * 16, out);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < G::kRotPer; ++k) {
        const int i = tid + k * kThreads;
        const uint4 partner = shfl_xor_u4(regs.r[k], G::HV);
        if (i < G::kRotItems) {
            const int row = i / G::kRotW, w = i % G::kRotW;
            const int64_t s = idx[row];
            if (s >= 0) {
                const int h = w / (2 * G::HV), v = w % (2 * G::HV);
                const bool first = v < G::HV;
                const int fb = (v % G::HV) * 8;
                bool patched = false;
                if (PATCH) {
                    patch_terms(*pa.pv, 1, pa.layer, pa.tok[row], pa.chunk[row],
                                h * G::kHalf * 2 + v * 8, add);
                    patched = pa.pv->u[1] != nullptr;
                }
                uint4 out;
                if (ident[row])
                    out = patched ? add_vec(regs.r[k], add) : regs.r[k];
                else if (IL)
                    out = rotate_vec_il<G>(regs.r[k], cs + row * cs_row_stride, v, add);
                else if (PACKED)
                    out = rotate_vec_packed(regs.r[k], partner, first,
                                            cs + row * cs_row_stride + fb / 8, G::HV);
                else
                    out = rotate_vec(regs.r[k], partner, first,
                                     cs + row * cs_row_stride + fb / 8, G::HV, add);
                st_stream(const_cast<char *>(at.rbase) + s * at.rstride + w * 16, out);
            }
        }
    }
}

} // namespace kvr
