// kv_patch_tc.cu -- the rank-m patch on the 5th-generation tensor cores
// (tcgen05), fused with the relocation (or applied in place).
//
// Kamera §2: KV^(B|A) = R(δ)·KV(B|∅) + U_m V_mᵀ.  For one (chunk, layer,
// channel) the patch is the product of U (rows x m) and V (cols x m)ᵀ, a
// dense contraction with a short inner dimension (m <= 16).  A block owns a
// slice of NB columns of one channel of one (chunk, layer) and walks the
// chunk in tiles of 128 rows.  Per tile:
//   * threads 0..127 each gather one row of the slice (NB x 2 bytes at its
//     source slot) into shared memory with a bulk copy (the TMA engine), so
//     the rows fly without occupying the load/store units;
//   * meanwhile the block converts the tile's U rows into bf16 high and low
//     parts (x ~ hi + lo to ~16 bits), stored as K-major core matrices
//     (8 rows x 16 B) once per slice; V's slice was split the same way once
//     per block; three tcgen05.mma kind::f16 (hi·hi, hi·lo, lo·hi)
//     accumulate the 128 x NB fp32 product in tensor memory;
//   * each thread is (row = tensor-memory lane, group of W columns = one
//     rotary head for the rotated channel, W = D), so it holds both halves
//     of every rotary pair it rewrites: it reads its part of the product 16
//     columns at a time with tcgen05.ld, forms rnd(R(δ)·x + patch) (rotated
//     channel) or rnd(x + patch) and writes it back into the tile;
//   * threads 0..127 write the rows to their target slots with bulk copies.
// The waits for copies and MMAs are bounded polls of mbarriers; tensor
// memory is released on every path.
#include <cuda_bf16.h>

#include "kv_launch.h"
#include "kv_tiles.cuh"

namespace kvr {
namespace tc {

constexpr int M = 128;                // rows per tile (MMA M)
constexpr int KP = 16;                // padded rank (MMA K for 16-bit inputs)
constexpr int A_BYTES = M * KP * 2;   // one of hi / lo
constexpr int64_t MMA_WAIT_NS = 1000000000ll;

// NB: columns per block (MMA N); W: columns per thread; D: rotary head dim of
// the rotated channel (D == W).  TILES row tiles of M rows are processed per
// step (each its own A operand and accumulator); a block's 128-thread parts
// split the columns (GROUPS = NB / W) or the row tiles, not both.
template <int NB_, int W_, int TILES_ = 1>
struct TcGeo {
    static constexpr int NB = NB_, W = W_, TILES = TILES_;
    static constexpr int GROUPS = NB / W;          // column groups per block
    static constexpr int ROWS = M * TILES;         // rows per step
    static constexpr int NT = M * GROUPS * TILES;  // threads per block
    static constexpr int B_BYTES = NB * KP * 2;    // one of hi / lo
    static constexpr int VECS = W * 2 / 16;        // 16-byte pieces of my columns
    static constexpr int HALF = W / 2;             // frequencies of my head
    static constexpr int TMEM_COLS = NB * TILES;   // accumulator columns
    static constexpr int MIN_BLOCKS = NT >= 256 ? 2 : (512 / NB < 4 ? 512 / NB : 4);
    static_assert(NB == 64 || NB == 128 || NB == 256, "MMA N");
    static_assert(W % 16 == 0 && NB % W == 0 && (GROUPS == 1 || GROUPS == 2), "groups");
    static_assert(GROUPS == 1 || TILES == 1, "split columns or rows, not both");
    static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
};

// Byte offset of element (r, k) in a K-major operand made of core matrices
// of 8 rows x 16 bytes: core matrices are 128 B apart along K and 256 B
// apart along M / N (the LBO / SBO of the descriptor below).
__device__ __forceinline__ uint32_t kmajor_off(int r, int k)
{
    return (uint32_t)((r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: no swizzle, LBO = 128 B, SBO = 256 B.
__device__ __forceinline__ uint64_t smem_desc(const void *p)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) |
           ((uint64_t)(256u >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
template <int N>
__device__ __forceinline__ constexpr uint32_t idesc()
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

template <int N>
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc<N>()), "r"(acc)
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.b32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait for an mbarrier phase (wall-time limit plus a poll cap).
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int64_t limit_ns)
{
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((int64_t)(global_ns() - t0) > limit_ns)
            return false;
    }
    return false;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Split 8 fp32 values (k .. k+7 of one row) into bf16 high / low parts and
// store them as one 16-byte core-matrix row each.
__device__ __forceinline__ void split_store8(const float *v, unsigned char *hi, unsigned char *lo)
{
    uint32_t h[4], w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * e]);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * e + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * e] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * e + 1] - __bfloat162float(h1));
        h[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        w[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    *reinterpret_cast<uint4 *>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Load 8 factor values (ranks k0 .. k0+7, zero past m) of one factor row.
__device__ __forceinline__ void load_factor8(const float *row, int k0, int m, float (&v)[8])
{
#pragma unroll
    for (int r = 0; r < 8; r += 4) {
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k0 + r < m)
            q = __ldg(reinterpret_cast<const float4 *>(row + k0 + r));
        v[r] = q.x;
        v[r + 1] = q.y;
        v[r + 2] = q.z;
        v[r + 3] = q.w;
    }
}

// Bulk (non-tensor) TMA copies of whole rows between global and shared
// memory; addresses and sizes are multiples of 16 bytes.
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"((uint32_t)__cvta_generic_to_shared(smem_src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Which blocks a launch covers: channels [ch0, ch0 + nch), `slices` slices
// of NB columns each; block x = (chunk * nch + ch - ch0) * slices + slice.
struct TcLaunch {
    int32_t ch0, nch, slices;
};

// Dynamic shared memory of one block: A (hi, lo) per row tile, B (hi, lo),
// then the rows of a step, ROWS rows of PITCH bytes.  The 16 spare bytes per row shift consecutive
// rows by four banks, so a warp reading the same piece of 32 rows is free of
// bank conflicts.
template <class G>
struct TcSmem {
    static constexpr int ROW_BYTES = G::NB * 2;
    static constexpr int PITCH = ROW_BYTES + 16;
    static constexpr int A_OFF = 0;                        // per row tile: hi, lo
    static constexpr int B_OFF = G::TILES * 2 * A_BYTES;
    static constexpr int X_OFF = B_OFF + 2 * G::B_BYTES;
    static constexpr int BYTES = X_OFF + G::ROWS * PITCH;
};

// A block owns NB columns of one channel of one (chunk, layer).  Per tile of
// 128 rows: threads 0..127 each gather one row with a bulk copy into shared
// memory while the block forms the A operand and the MMAs run; then every
// thread rewrites its (row, column group) of the tile in shared memory and
// threads 0..127 write the rows back with bulk copies.
template <class G, bool RELOC>
__device__ __forceinline__ void patch_tc_body(const RelocParams &p, const TcLaunch &tl,
                                              const int bx)
{
    using S = TcSmem<G>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *b_hi = smem + S::B_OFF, *b_lo = b_hi + G::B_BYTES;
    unsigned char *xs = smem + S::X_OFF;
    // cos/sin per pair of frequencies k = (2k, 2k+1): cs_c[k] = (c1, c1', c2, c2'),
    // cs_s[k] = (s1, s1', s2, s2'); cos = c1 + c2, sin = s1 + s2
    __shared__ __align__(16) float cs_c[G::HALF * 2], cs_s[G::HALF * 2];
    __shared__ __align__(8) uint64_t s_bar[2]; // [0] rows landed, [1] MMAs done
    __shared__ uint32_t s_tmem;
    __shared__ int32_t s_ok;

    if (gate_closed(p.gate))
        return; // a debug check found an overlap: store nothing
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per_chunk = tl.nch * tl.slices;
    const int c = bx / per_chunk, l = blockIdx.y;
    const int ch = tl.ch0 + (bx / tl.slices) % tl.nch;
    const int col0 = (bx % tl.slices) * G::NB;
    if (bx == 0 && l == 0 && tid == 0) {
        if (p.tok_off[0] != 0 || p.tok_off[p.num_chunks] != p.total_tokens)
            set_status(p.status, kStatusOutOfRange);
    }
    const bool patched = p.patch.u[ch] != nullptr;
    if (!RELOC && !patched)
        return; // in place and nothing to add: the rows stay as they are
    const int64_t t0 = p.tok_off[c];
    const int64_t n = max((int64_t)0, (int64_t)p.tok_off[c + 1] - t0);
    // U row of the chunk's first token: call order, or the caller's map
    const int64_t u0 = p.patch.u_chunk_tok ? p.patch.u_chunk_tok[c] : t0;
    if (patched) {
        // the chunk's U rows and V slot must lie inside the stated extents
        const int64_t vs = p.patch.v_chunk ? p.patch.v_chunk[c] : c;
        if (n > 0 && !(patch_rows_ok(p.patch, u0, vs) && patch_rows_ok(p.patch, u0 + n - 1, vs))) {
            if (tid == 0)
                set_status(p.status, kStatusOutOfRange);
            return; // block-uniform: nothing allocated yet
        }
    }
    const int32_t req = p.chunk_req[c];
    const bool req_ok = req >= 0 && req < p.num_reqs;
    const int32_t *bt = p.block_tables + (int64_t)(req_ok ? req : 0) * p.max_blocks;
    const int64_t pos0 = p.chunk_dst_pos[c];
    const bool rotate = RELOC && ch == 1 && p.delta[c] != 0;
    const int m = p.patch.m;
    const bool owner = tid < G::ROWS;           // gathers / writes back row `tid`
    const int lane_row = (warp & 3) * 32 + lane; // my TMEM lane
    const int part = warp >> 2;                  // my 128-thread part of the block
    const int rt = G::TILES > 1 ? part : 0;      // my row tile
    const int grp = G::TILES > 1 ? 0 : part;     // my column group
    const int row = rt * M + lane_row;           // my row in the rewrite
    const int cg = grp * G::W;
    const PoolView &sp = RELOC ? p.src : p.dst;
    const char *src_base = (ch == 0 ? sp.copy + (int64_t)l * sp.copy_ls
                                    : sp.rot + (int64_t)l * sp.rot_ls) + col0 * 2;
    const int64_t src_ss = ch == 0 ? sp.copy_ss : sp.rot_ss;
    char *dst_base = (ch == 0 ? p.dst.copy + (int64_t)l * p.dst.copy_ls
                              : p.dst.rot + (int64_t)l * p.dst.rot_ls) + col0 * 2;
    const int64_t dst_ss = ch == 0 ? p.dst.copy_ss : p.dst.rot_ss;

    // --- once per block: V's slice as the B operand, cos/sin, barriers, TMEM
    if (patched) {
        const int64_t vslot = p.patch.v_chunk ? p.patch.v_chunk[c] : c;
        const float *vb = p.patch.v[ch] + (int64_t)l * p.patch.v_ls[ch] +
                          vslot * p.patch.v_cs[ch] + (int64_t)col0 * p.patch.v_cols[ch];
        for (int i = tid; i < G::NB * 2; i += G::NT) {
            const int nn = i >> 1, k0 = (i & 1) * 8;
            float v[8];
            load_factor8(vb + (int64_t)nn * p.patch.v_cols[ch], k0, m, v);
            split_store8(v, b_hi + kmajor_off(nn, k0), b_lo + kmajor_off(nn, k0));
        }
    }
    if (rotate && tid < G::HALF) {
        const float4 q = p.table[(int64_t)c * G::HALF + tid];
        const int at = (tid >> 1) * 4 + (tid & 1);
        cs_c[at] = q.x;
        cs_c[at + 2] = q.y;
        cs_s[at] = q.z;
        cs_s[at + 2] = q.w;
    }
    const uint32_t bar_x = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    const uint32_t bar_mma = (uint32_t)__cvta_generic_to_shared(&s_bar[1]);
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar_x), "r"(G::ROWS)
                     : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_mma) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_ok = 1;
    }
    if (patched && warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(&s_tmem)),
                     "r"((uint32_t)G::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = patched ? s_tmem : 0u;
    const uint32_t t_row =
        tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(rt * G::NB + cg);

    // slots of row `tid` of tile t (owners only); a bad index is reported and
    // its row skipped
    auto row_slots = [&](int64_t t, int64_t &src, int64_t &dst) {
        const int64_t i = t * G::ROWS + tid;
        src = dst = -1;
        if (i >= n)
            return;
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
    };

    const int64_t ntiles = (n + G::ROWS - 1) / G::ROWS;
    unsigned char *my_row = xs + tid * S::PITCH;                   // owner's row
    unsigned char *xr = xs + row * S::PITCH + cg * 2;              // my part in the rewrite
    uint4 *xq = reinterpret_cast<uint4 *>(xr);
    int64_t src = -1, dst = -1;
    if (owner && ntiles > 0)
        row_slots(0, src, dst);
    uint32_t ph_x = 0, ph_mma = 0;
    // U rows of a tile for the A operand, one or two (row, 8 ranks) items per thread
    constexpr int kUItems = (G::ROWS * 2 + G::NT - 1) / G::NT;
    float u_next[kUItems][8];
    auto load_u = [&](int64_t t) {
#pragma unroll
        for (int it = 0; it < kUItems; ++it) {
            const int e = tid + it * G::NT;
            const int r = e >> 1, k0 = (e & 1) * 8;
            const int64_t i = t * G::ROWS + r;
            if (e < G::ROWS * 2 && i < n) {
                load_factor8(p.patch.u[ch] + (int64_t)l * p.patch.u_ls[ch] +
                                 (u0 + i) * p.patch.u_ts[ch],
                             k0, m, u_next[it]);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    u_next[it][q] = 0.0f;
            }
        }
    };
    for (int64_t t = 0; t < ntiles; ++t) {
        int64_t my_dst = -1;
        if (owner) {
            // the previous tile's write-back has finished reading this row
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            if (src >= 0) {
                mbar_arrive_tx(bar_x, S::ROW_BYTES);
                bulk_load(my_row, src_base + src * src_ss, S::ROW_BYTES, bar_x);
            } else {
                mbar_arrive(bar_x);
            }
            my_dst = dst;
            if (t + 1 < ntiles) // the next tile's slots, while this one is in flight
                row_slots(t + 1, src, dst);
        }
        if (patched) {
            // A operand: the tile's U rows (fetched during the previous tile's
            // rewrite) split into bf16 hi / lo (zero past the chunk)
            if (t == 0)
                load_u(t);
#pragma unroll
            for (int it = 0; it < kUItems; ++it) {
                const int e = tid + it * G::NT;
                if (e < G::ROWS * 2) {
                    const int r = e >> 1, k0 = (e & 1) * 8;
                    unsigned char *a_hi = smem + S::A_OFF + (r / M) * 2 * A_BYTES;
                    unsigned char *a_lo = a_hi + A_BYTES;
                    split_store8(u_next[it], a_hi + kmajor_off(r % M, k0),
                                 a_lo + kmajor_off(r % M, k0));
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            fence_before();
            __syncthreads(); // A complete; the previous tile's accumulator reads are done
            if (tid == 0) {
                fence_after();
#pragma unroll
                for (int q = 0; q < G::TILES; ++q) {
                    const unsigned char *a_hi = smem + S::A_OFF + q * 2 * A_BYTES;
                    const unsigned char *a_lo = a_hi + A_BYTES;
                    const uint32_t d = tmem + (uint32_t)(q * G::NB);
                    mma_bf16<G::NB>(d, smem_desc(a_hi), smem_desc(b_hi), 0u);
                    mma_bf16<G::NB>(d, smem_desc(a_hi), smem_desc(b_lo), 1u);
                    mma_bf16<G::NB>(d, smem_desc(a_lo), smem_desc(b_hi), 1u);
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_mma)
                             : "memory");
                if (!mbar_wait(bar_mma, ph_mma, MMA_WAIT_NS)) {
                    set_status(p.status, kStatusTimeout);
                    mbar_wait(bar_mma, ph_mma, MMA_WAIT_NS); // once more before memory is released
                    s_ok = 0;
                }
            }
            ph_mma ^= 1u;
        }
        if (!mbar_wait(bar_x, ph_x, MMA_WAIT_NS)) {
            set_status(p.status, kStatusTimeout);
            mbar_wait(bar_x, ph_x, MMA_WAIT_NS); // the copies in flight, once more
            s_ok = 0;
        }
        ph_x ^= 1u;
        __syncthreads();
        fence_after();
        if (!s_ok)
            break;
        if (patched && t + 1 < ntiles)
            load_u(t + 1); // lands while this tile is rewritten

        // rewrite my (row, column group) of the tile in place; a warp whose 32
        // rows all lie past the chunk's end has nothing to rewrite
        const bool warp_rows = t * G::ROWS + rt * M + (warp & 3) * 32 < n;
        if (!warp_rows) {
        } else if (patched && rotate) {
            const ulonglong2 *cc = reinterpret_cast<const ulonglong2 *>(cs_c);
            const ulonglong2 *ss = reinterpret_cast<const ulonglong2 *>(cs_s);
            // one 16-frequency group at a time: the registers this leaves free
            // hold the next tile's U rows
#pragma unroll 1
            for (int f0 = 0; f0 < G::HALF; f0 += 16) {
                uint32_t a1[16], a2[16];
                tmem_ld16(t_row + (uint32_t)f0, a1);
                tmem_ld16(t_row + (uint32_t)(f0 + G::HALF), a2);
                const uint4 p0 = xq[f0 / 8], p1 = xq[f0 / 8 + 1];
                const uint4 q0 = xq[(f0 + G::HALF) / 8], q1 = xq[(f0 + G::HALF) / 8 + 1];
                const uint32_t w1s[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                const uint32_t w2s[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                uint32_t o1[8], o2[8];
                f2 chk = 0ull;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    // frequencies f0+2k, f0+2k+1 at once: (x1, x2) = (x[j], x[j+D/2])
                    // turned by δθ_j, with c1, s1 short enough for exact products
                    const ulonglong2 C = cc[f0 / 2 + k], S = ss[f0 / 2 + k];
                    const f2 x1 = f2_of_bf16x2(w1s[k]), x2 = f2_of_bf16x2(w2s[k]);
                    const f2 x2n = f2_of_bf16x2(w2s[k] ^ 0x80008000u);
                    const f2 r1 = f2_add(f2_fma(x1, C.x, f2_mul(x2n, S.x)),
                                         f2_add(f2_fma(x1, C.y, f2_mul(x2n, S.y)),
                                                f2_of_bits(a1[2 * k], a1[2 * k + 1])));
                    const f2 r2 = f2_add(f2_fma(x2, C.x, f2_mul(x1, S.x)),
                                         f2_add(f2_fma(x2, C.y, f2_mul(x1, S.y)),
                                                f2_of_bits(a2[2 * k], a2[2 * k + 1])));
                    chk = f2_fma(r1, 0ull, chk); // NaN if any result is Inf or NaN
                    chk = f2_fma(r2, 0ull, chk);
                    o1[k] = bf16x2_rne(r1);
                    o2[k] = bf16x2_rne(r2);
                }
                if (__any_sync(0xFFFFFFFFu, f2_has_nan(chk))) {
                    // Inf / NaN in the block (rare; whole warp, inputs read
                    // again): elements with a non-finite input take plain
                    // IEEE arithmetic, as the fp64 definition does
                    uint32_t b1[16], b2[16];
                    tmem_ld16(t_row + (uint32_t)f0, b1);
                    tmem_ld16(t_row + (uint32_t)(f0 + G::HALF), b2);
                    const uint16_t *x1h = reinterpret_cast<const uint16_t *>(xq) + f0;
                    const uint16_t *x2h = x1h + G::HALF;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t h1 = x1h[e], h2 = x2h[e];
                        if (bf16_finite(h1) && bf16_finite(h2))
                            continue;
                        const int at = ((f0 + e) >> 1) * 4 + (e & 1);
                        const float cs = cs_c[at] + cs_c[at + 2], sn = cs_s[at] + cs_s[at + 2];
                        const float x1 = __uint_as_float(h1 << 16), x2 = __uint_as_float(h2 << 16);
                        const uint32_t y1 = bf16_rne((x1 * cs - x2 * sn) + __uint_as_float(b1[e]));
                        const uint32_t y2 = bf16_rne((x1 * sn + x2 * cs) + __uint_as_float(b2[e]));
                        const int sh = 16 * (e & 1);
                        o1[e >> 1] = (o1[e >> 1] & ~(0xFFFFu << sh)) | (y1 << sh);
                        o2[e >> 1] = (o2[e >> 1] & ~(0xFFFFu << sh)) | (y2 << sh);
                    }
                }
                xq[f0 / 8] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                xq[f0 / 8 + 1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
                xq[(f0 + G::HALF) / 8] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                xq[(f0 + G::HALF) / 8 + 1] = make_uint4(o2[4], o2[5], o2[6], o2[7]);
            }
        } else if (patched) {
#pragma unroll
            for (int c16 = 0; c16 < G::W; c16 += 16) {
                uint32_t a[16];
                tmem_ld16(t_row + (uint32_t)c16, a);
                const uint4 p0 = xq[c16 / 8], p1 = xq[c16 / 8 + 1];
                const uint32_t ws[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                uint32_t o[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    o[k] = bf16x2_rne(f2_add(f2_of_bf16x2(ws[k]),
                                             f2_of_bits(a[2 * k], a[2 * k + 1])));
                xq[c16 / 8] = make_uint4(o[0], o[1], o[2], o[3]);
                xq[c16 / 8 + 1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        } else if (rotate) {
            // no factors on this channel: the correctly rounded rotation of
            // the unpatched relocation (the verbatim part needs no rewrite)
#pragma unroll
            for (int f0 = 0; f0 < G::HALF; f0 += 8) {
                const uint4 pa = xq[f0 / 8], pb = xq[(f0 + G::HALF) / 8];
                const uint32_t w1s[4] = {pa.x, pa.y, pa.z, pa.w};
                const uint32_t w2s[4] = {pb.x, pb.y, pb.z, pb.w};
                uint32_t o1[4], o2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t w1 = w1s[e], w2 = w2s[e];
                    const int at = ((f0 + 2 * e) >> 1) * 4;
                    const float4 c0 = make_float4(cs_c[at], cs_c[at + 2], cs_s[at], cs_s[at + 2]);
                    const float4 c1 =
                        make_float4(cs_c[at + 1], cs_c[at + 3], cs_s[at + 1], cs_s[at + 3]);
                    o1[e] = rotate_one(w1 & 0xFFFFu, w2 & 0xFFFFu, c0, true, 0.0f) |
                            (rotate_one(w1 >> 16, w2 >> 16, c1, true, 0.0f) << 16);
                    o2[e] = rotate_one(w1 & 0xFFFFu, w2 & 0xFFFFu, c0, false, 0.0f) |
                            (rotate_one(w1 >> 16, w2 >> 16, c1, false, 0.0f) << 16);
                }
                xq[f0 / 8] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                xq[(f0 + G::HALF) / 8] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
            }
        }
        // generic-proxy writes of the tile become visible to the bulk copies
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        fence_before();
        __syncthreads();
        if (owner && my_dst >= 0)
            bulk_store(dst_base + my_dst * dst_ss, my_row, S::ROW_BYTES);
    }
    if (owner)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    fence_before();
    __syncthreads();
    if (patched && warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)G::TMEM_COLS)
                     : "memory");
}

template <class G, bool RELOC>
__global__ void __launch_bounds__(G::NT, G::MIN_BLOCKS)
patch_tc_kernel(const __grid_constant__ RelocParams p, const TcLaunch tl)
{
    patch_tc_body<G, RELOC>(p, tl, (int)blockIdx.x);
}

// MLA rows in one launch: the first n_kv blocks take the latent c_KV in
// slices of 256 columns (GA), the others the 64-column k_pe in two row tiles
// per step (GB), so the small k_pe blocks run alongside the c_KV traffic.
using GeoMlaKv = TcGeo<256, 128>;
using GeoMlaPe = TcGeo<64, 64, 2>;
static_assert(GeoMlaKv::NT == GeoMlaPe::NT, "one block shape");

// Blocks 3c, 3c+1: chunk c's two c_KV slices; block 3c+2: its k_pe.
template <bool RELOC>
__global__ void __launch_bounds__(GeoMlaKv::NT, 2)
patch_tc_mla_kernel(const __grid_constant__ RelocParams p)
{
    const int c = (int)blockIdx.x / 3, j = (int)blockIdx.x % 3;
    if (j < 2)
        patch_tc_body<GeoMlaKv, RELOC>(p, TcLaunch{0, 1, 2}, 2 * c + j);
    else
        patch_tc_body<GeoMlaPe, RELOC>(p, TcLaunch{1, 1, 1}, c);
}

static cudaError_t launch_mla(const RelocParams &p, cudaStream_t stream)
{
    const int64_t blocks = (int64_t)p.num_chunks * 3;
    if (blocks > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks, (unsigned)p.src.num_layers);
    constexpr int smem = TcSmem<GeoMlaKv>::BYTES > TcSmem<GeoMlaPe>::BYTES
                             ? TcSmem<GeoMlaKv>::BYTES
                             : TcSmem<GeoMlaPe>::BYTES;
    return with_bool(p.in_place == 0, [&](auto reloc) {
        constexpr bool R = decltype(reloc)::value;
        cudaError_t e = cudaFuncSetAttribute(patch_tc_mla_kernel<R>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        patch_tc_mla_kernel<R><<<grid, GeoMlaKv::NT, smem, stream>>>(p);
        return cudaGetLastError();
    });
}

template <class G>
static cudaError_t launch_geo(const RelocParams &p, TcLaunch tl, cudaStream_t stream)
{
    const int64_t blocks = (int64_t)p.num_chunks * tl.nch * tl.slices;
    if (blocks == 0)
        return cudaSuccess;
    if (blocks > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks, (unsigned)p.src.num_layers);
    constexpr int smem = TcSmem<G>::BYTES;
    cudaError_t e;
    if (p.in_place) {
        if ((e = cudaFuncSetAttribute(patch_tc_kernel<G, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return e;
        patch_tc_kernel<G, false><<<grid, G::NT, smem, stream>>>(p, tl);
    } else {
        if ((e = cudaFuncSetAttribute(patch_tc_kernel<G, true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return e;
        patch_tc_kernel<G, true><<<grid, G::NT, smem, stream>>>(p, tl);
    }
    return cudaGetLastError();
}

} // namespace tc

bool patch_tc_supported(const RelocParams &p, RowKind kind)
{
    (void)kind;
    // the epilogue turns rotate-half pairs; relocations of interleaved rows
    // take the token-tiled kernel (an in-place patch rotates nothing)
    return p.patched && p.patch.m <= tc::KP && p.src.num_layers <= 65535 &&
           (p.in_place || !p.dst.il);
}

int patch_tc_launches(const RelocParams &p, RowKind kind)
{
    return (kind == RowKind::Mla && p.in_place) ? 2 : 1;
}

cudaError_t launch_patch_tc(const RelocParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.num_chunks == 0)
        return cudaSuccess;
    if (kind != RowKind::Mla) {
        // K and V rows of H heads of 128: H / 2 slices of two heads per channel
        const int32_t slices = kind == RowKind::Gqa ? 4 : kind == RowKind::Gqa4 ? 2 : 16;
        return tc::launch_geo<tc::TcGeo<256, 128>>(p, tc::TcLaunch{0, 2, slices}, stream);
    }
    // MLA relocation: the 512-wide latent as 2 slices of 256 and the 64-wide
    // k_pe in one launch, so the k_pe blocks run alongside the c_KV traffic.
    // In place (no gather, no rotation) the k_pe rows are light enough that a
    // launch of their own, four blocks per SM, is faster.
    if (!p.in_place)
        return tc::launch_mla(p, stream);
    cudaError_t e = tc::launch_geo<tc::TcGeo<256, 128>>(p, tc::TcLaunch{0, 1, 2}, stream);
    if (e != cudaSuccess)
        return e;
    return tc::launch_geo<tc::TcGeo<64, 64>>(p, tc::TcLaunch{1, 1, 1}, stream);
}

} // namespace kvr
