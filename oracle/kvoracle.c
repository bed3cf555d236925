/*
 * kvoracle.c -- plain, slow, fp64 CPU oracle for KV relocation, splice and patch.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product path
 * (the CUDA library) never calls, links or includes anything from here, and
 * this file includes nothing from the product.
 *
 * What it computes, and where the pages define it (gist.science summaries):
 *   - Leyline: KV-Cache Directives for Agentic Inference
 *       §2.1  directive D = (s_start, s_end, R, m), modes AMORTIZE / FORGET
 *       §2.2  Δ = |R| - |S|;  K_pe_new[i] = R(Δ)·K_pe[i];  R(a)R(b) = R(a+b);
 *             K_nope and V (for MLA: the latent c_KV) are kept as they are
 *       §2.3  the rotation is applied to the K_pe band of every downstream
 *             slot, which is re-indexed
 *       §4.3  rotation math in higher precision, KV stored in bf16
 *   - Irminsul: MLA-native position-independent cache
 *       §2.1  cKV (512 dims) is reused verbatim, k_r (64 dims) is rotated
 *       §2.2  δ = p_target - p_source, R(δ) applied to the stored k_r
 *   - Kamera: unified, position-invariant multimodal KV cache
 *       §2    KV^(B|A) = R(δ)·KV(B|∅) + U_m V_mᵀ; GQA re-rotates the whole K
 *             and patches K and V; MLA rotates only k_rope, reuses c_KV byte
 *             for byte and patches both channels
 *
 * Readings where the pages are silent (each is used below and nowhere else):
 *   - RoPE pairs are "rotate-half": on a d-dim rotary vector, pair j is
 *     (x[j], x[j+d/2]) for j < d/2, with frequency θ_j = base^(-2j/d).
 *   - R(δ) turns pair j by the angle δ·θ_j in the positive sense:
 *       y[j] = x[j]cos - x[j+h]sin,  y[j+h] = x[j]sin + x[j+h]cos,
 *     so that R(δ) applied to a key encoded at position p equals the key
 *     encoded at p + δ.
 *   - Spans are half open: S = [s_start, s_end), |S| = s_end - s_start.
 *   - Stub rows (the prefilled replacement R) are written verbatim at their
 *     final positions; they are not rotated.
 *   - Rounding is one direct fp64 -> bf16 round-to-nearest-even per stored
 *     value (no detour through fp32).
 *   - The rank-m patch is added after the rotation, in the target frame; in
 *     a fused relocation the unrounded rotated value receives the patch and
 *     the sum is rounded once.
 *
 * Memory layout used by the oracle (its own, independent of the library's):
 *   copy part  [L][slots][copy_dim]            bf16 bit patterns (uint16)
 *   rot part   [L][slots][rot_heads*rot_d]     bf16 bit patterns (uint16)
 *   slot of logical position p of request q:  bt[q][p / B] * B + p % B
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (see build.py).
 * Contraction is off so that x*c - y*s rounds each product, on x86 and Arm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVO_OK 0
#define KVO_ERR_INVALID 1
#define KVO_ERR_RANGE 2
#define KVO_ERR_CAPACITY 3

/* ------------------------------------------------------------------ */
/* bf16 <-> fp64                                                        */
/* ------------------------------------------------------------------ */

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
double kvo_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, in one step.  Finite results are n * 2^q with n an
 * integer and q the exponent of the bf16 unit in the last place:
 *   |v| in [2^E, 2^(E+1)),  E >= -126  ->  q = E - 7
 *   |v| <  2^-126 (subnormal range)    ->  q = -133
 * The scaling by 2^-q is exact, rint() in the default rounding mode breaks
 * ties to even, and anything above the largest finite bf16 becomes infinity. */
uint16_t kvo_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
    int E = e - 1;
    if (E < -126)
        E = -126;
    int q = E - 7;
    double n = rint(ldexp(a, -q));
    double r = ldexp(n, q);
    if (r > ldexp(255.0, 120)) /* largest finite bf16 = (2^8 - 1) * 2^120 */
        return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* Element-wise versions of the two conversions above. */
void kvo_round_bf16_n(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_round_bf16(v[i]);
}

void kvo_bf16_to_f64_n(const uint16_t *b, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_bf16_to_f64(b[i]);
}

/* ------------------------------------------------------------------ */
/* The rotation R(δ) on one rotary vector                               */
/* ------------------------------------------------------------------ */

/* Frequency of pair j of a d-dim rotary vector: θ_j = base^(-2j/d). */
double kvo_theta(double base, int j, int d)
{
    return pow(base, -2.0 * (double)j / (double)d);
}

/* y = R(δ)·x in fp64, unrounded.  x and y may alias.  Leyline §2.2,
 * Irminsul §2.2: one 2x2 rotation per frequency pair. */
void kvo_rotate_f64(const double *x, double *y, int d, int64_t delta, double base)
{
    int h = d / 2;
    for (int j = 0; j < h; ++j) {
        double a = (double)delta * kvo_theta(base, j, d);
        double c = cos(a), s = sin(a);
        double lo = x[j], hi = x[j + h];
        y[j] = lo * c - hi * s;
        y[j + h] = lo * s + hi * c;
    }
}

/* The same rotation with the interleaved pairing that some models store
 * k_pe in: pair j is (x[2j], x[2j+1]), with the same θ_j. */
void kvo_rotate_f64_il(const double *x, double *y, int d, int64_t delta, double base)
{
    for (int j = 0; j < d / 2; ++j) {
        double a = (double)delta * kvo_theta(base, j, d);
        double c = cos(a), s = sin(a);
        double even = x[2 * j], odd = x[2 * j + 1];
        y[2 * j] = even * c - odd * s;
        y[2 * j + 1] = even * s + odd * c;
    }
}

/* y_exact = R(δ)·x in fp64 for a bf16 vector x (not rounded); `il` selects
 * the interleaved pairing. */
static void rotate_bf16_exact(const uint16_t *x, double *y, int d, int64_t delta, double base,
                              int il)
{
    for (int i = 0; i < d; ++i)
        y[i] = kvo_bf16_to_f64(x[i]);
    if (il)
        kvo_rotate_f64_il(y, y, d, delta, base);
    else
        kvo_rotate_f64(y, y, d, delta, base);
}

static void rotate_bf16_pairs(const uint16_t *x, uint16_t *y, int d, int64_t delta, double base,
                              int il)
{
    if (delta == 0) {
        memmove(y, x, (size_t)d * sizeof *y);
        return;
    }
    double t[1024];
    rotate_bf16_exact(x, t, d, delta, base, il);
    for (int i = 0; i < d; ++i)
        y[i] = kvo_round_bf16(t[i]);
}

/* y = rnd(R(δ)·x) on bf16 vectors.  R(0) is the identity, bit for bit
 * (this also fixes the sign of zeros).  x and y may alias. */
void kvo_rotate_bf16(const uint16_t *x, uint16_t *y, int d, int64_t delta, double base)
{
    rotate_bf16_pairs(x, y, d, delta, base, 0);
}

/* The same with the interleaved pairing. */
void kvo_rotate_bf16_il(const uint16_t *x, uint16_t *y, int d, int64_t delta, double base)
{
    rotate_bf16_pairs(x, y, d, delta, base, 1);
}

/* ------------------------------------------------------------------ */
/* Pool geometry                                                       */
/* ------------------------------------------------------------------ */

typedef struct {
    int num_layers;      /* L */
    int64_t num_slots;   /* slots per layer */
    int block_size;      /* B: tokens per paged block */
    int copy_dim;        /* verbatim part: c_KV (512) or GQA V (H*D) */
    int rot_heads;       /* 1 for MLA k_pe, H for GQA K */
    int rot_d;           /* rotary dim per head: 64 (MLA) or 128 (GQA) */
    double rope_base;    /* 10000, 500000, ... */
    uint16_t *copy;      /* [L][num_slots][copy_dim] */
    uint16_t *rot;       /* [L][num_slots][rot_heads*rot_d] */
    int pair_convention; /* 0: rotate-half (x[j], x[j+d/2]); 1: interleaved (x[2j], x[2j+1]) */
} kvo_pool;

/* Rank-m patch factors (Kamera §2: U_m V_mᵀ), one pair per channel.
 * Channel 0 is the verbatim part, channel 1 the rotated part.  A NULL u or v
 * means no patch on that channel.
 *   U[ch](l, t, r)      = u[ch][l*u_layer_stride[ch] + t*u_tok_stride[ch] + r]
 *   V[ch](l, c, col, r) = v[ch][l*v_layer_stride[ch] + c*v_chunk_stride[ch]
 *                              + col*v_col_stride[ch] + r]
 * t is the token's U row and c the chunk's V slot; col is the column inside
 * the channel (for the rotated part: head*rot_d + element).  By default t is
 * the token's index in the call's token list (the chunk's first token index
 * plus its offset in the chunk) and c the chunk's index in the call.  Factors
 * kept once per canonical chunk and reused by any later call (Kamera's
 * reorder with one orbit patch, recall of an evicted chunk) are addressed
 * through the optional per-chunk maps instead:
 *   u_chunk_tok[c]  U row of chunk c's first token (its tokens follow it),
 *   v_chunk[c]      V slot of chunk c,
 * both for both channels; the caller keeps them inside the factor arrays. */
typedef struct {
    int m;
    const float *u[2];
    int64_t u_layer_stride[2], u_tok_stride[2];
    const float *v[2];
    int64_t v_layer_stride[2], v_chunk_stride[2], v_col_stride[2];
    const int64_t *u_chunk_tok; /* NULL: the call's token order */
    const int32_t *v_chunk;     /* NULL: the call's chunk order */
} kvo_patch;

static int rot_width(const kvo_pool *p) { return p->rot_heads * p->rot_d; }

static uint16_t *copy_row(const kvo_pool *p, int l, int64_t slot)
{
    return p->copy + ((int64_t)l * p->num_slots + slot) * p->copy_dim;
}

static uint16_t *rot_row(const kvo_pool *p, int l, int64_t slot)
{
    return p->rot + ((int64_t)l * p->num_slots + slot) * rot_width(p);
}

static int pool_ok(const kvo_pool *p)
{
    return p && p->copy && p->rot && p->num_layers > 0 && p->num_slots > 0 &&
           p->block_size > 0 && p->copy_dim >= 0 && p->rot_heads > 0 &&
           p->rot_d > 0 && p->rot_d % 2 == 0 && p->rot_d <= 1024 &&
           p->num_slots % p->block_size == 0 && p->rope_base > 0.0 &&
           (p->pair_convention == 0 || p->pair_convention == 1);
}

/* Physical slot of logical position pos in the block table row bt_row, or -1
 * if the position lies outside the table or the block id is not in the pool. */
static int64_t slot_of(const kvo_pool *p, const int32_t *bt_row, int max_blocks, int64_t pos)
{
    if (pos < 0)
        return -1;
    int64_t b = pos / p->block_size;
    if (b >= max_blocks)
        return -1;
    int64_t blk = bt_row[b];
    if (blk < 0 || blk >= p->num_slots / p->block_size)
        return -1;
    return blk * p->block_size + pos % p->block_size;
}

/* Σ_r U(l,t,r)·V(l,c,col,r) for one channel, in fp64, r ascending. */
/* U row of the call's token t (of chunk c) and V slot of chunk c. */
static int64_t u_row(const kvo_patch *pt, const int32_t *tok_off, int64_t c, int64_t t)
{
    return pt->u_chunk_tok ? pt->u_chunk_tok[c] + (t - tok_off[c]) : t;
}

static int64_t v_slot(const kvo_patch *pt, int64_t c) { return pt->v_chunk ? pt->v_chunk[c] : c; }

static double patch_term(const kvo_patch *pt, int ch, int l, int64_t t, int64_t c, int col)
{
    const float *u = pt->u[ch] + l * pt->u_layer_stride[ch] + t * pt->u_tok_stride[ch];
    const float *v = pt->v[ch] + l * pt->v_layer_stride[ch] + c * pt->v_chunk_stride[ch] +
                     (int64_t)col * pt->v_col_stride[ch];
    double s = 0.0;
    for (int r = 0; r < pt->m; ++r)
        s += (double)u[r] * (double)v[r];
    return s;
}

static int has_patch(const kvo_patch *pt, int ch)
{
    return pt && pt->m > 0 && pt->u[ch] && pt->v[ch];
}

/* ------------------------------------------------------------------ */
/* Relocation (Irminsul §2.2, Kamera §2)                                */
/* ------------------------------------------------------------------ */

/* For each chunk c, layer l and token i of the chunk:
 *   t    = tok_off[c] + i                    (index into src_slots)
 *   pos  = chunk_dst_pos[c] + i              (logical target position)
 *   dst  = slot of pos in block table row chunk_req[c]
 *   copy part:  dst row = src row, byte for byte
 *   rot part:   each head rotated by R(delta[c]), rounded to bf16
 * With a patch, each channel's value becomes rnd(x + Σ_r U·V), where x is
 * the copied value (copy part) or the unrounded rotated value (rot part).
 * All indices are checked first; on any bad index nothing is written and
 * KVO_ERR_RANGE is returned. */
int kvo_relocate(const kvo_pool *src, kvo_pool *dst, int num_chunks, const int32_t *tok_off,
                 const int32_t *src_slots, const int32_t *chunk_req, const int32_t *chunk_dst_pos,
                 const int32_t *delta, const int32_t *block_tables, int num_reqs, int max_blocks,
                 const kvo_patch *patch)
{
    if (!pool_ok(src) || !pool_ok(dst) || num_chunks < 0)
        return KVO_ERR_INVALID;
    if (src->num_layers != dst->num_layers || src->copy_dim != dst->copy_dim ||
        src->rot_heads != dst->rot_heads || src->rot_d != dst->rot_d ||
        src->rope_base != dst->rope_base || src->pair_convention != dst->pair_convention)
        return KVO_ERR_INVALID;
    if (tok_off[0] != 0)
        return KVO_ERR_INVALID;
    for (int c = 0; c < num_chunks; ++c) {
        if (tok_off[c + 1] < tok_off[c])
            return KVO_ERR_INVALID;
        if (chunk_req[c] < 0 || chunk_req[c] >= num_reqs)
            return KVO_ERR_RANGE;
        const int32_t *bt = block_tables + (int64_t)chunk_req[c] * max_blocks;
        for (int64_t t = tok_off[c]; t < tok_off[c + 1]; ++t) {
            if (src_slots[t] < 0 || src_slots[t] >= src->num_slots)
                return KVO_ERR_RANGE;
            if (slot_of(dst, bt, max_blocks, chunk_dst_pos[c] + (t - tok_off[c])) < 0)
                return KVO_ERR_RANGE;
        }
    }
    const int L = src->num_layers, cd = src->copy_dim, rd = src->rot_d, rh = src->rot_heads;
    double ex[1024];
    for (int c = 0; c < num_chunks; ++c) {
        const int32_t *bt = block_tables + (int64_t)chunk_req[c] * max_blocks;
        for (int l = 0; l < L; ++l) {
            for (int64_t t = tok_off[c]; t < tok_off[c + 1]; ++t) {
                int64_t s = src_slots[t];
                int64_t d = slot_of(dst, bt, max_blocks, chunk_dst_pos[c] + (t - tok_off[c]));
                const uint16_t *sc = copy_row(src, l, s);
                const uint16_t *sr = rot_row(src, l, s);
                uint16_t *dc = copy_row(dst, l, d);
                uint16_t *dr = rot_row(dst, l, d);
                if (has_patch(patch, 0)) {
                    for (int col = 0; col < cd; ++col)
                        dc[col] = kvo_round_bf16(kvo_bf16_to_f64(sc[col]) +
                                                 patch_term(patch, 0, l,
                                                            u_row(patch, tok_off, c, t),
                                                            v_slot(patch, c), col));
                } else {
                    memcpy(dc, sc, (size_t)cd * sizeof *dc);
                }
                for (int h = 0; h < rh; ++h) {
                    if (has_patch(patch, 1)) {
                        if (delta[c] == 0) {
                            for (int i = 0; i < rd; ++i)
                                ex[i] = kvo_bf16_to_f64(sr[h * rd + i]);
                        } else {
                            rotate_bf16_exact(sr + h * rd, ex, rd, delta[c], src->rope_base,
                                              src->pair_convention);
                        }
                        for (int i = 0; i < rd; ++i)
                            dr[h * rd + i] =
                                kvo_round_bf16(ex[i] + patch_term(patch, 1, l,
                                                                  u_row(patch, tok_off, c, t),
                                                                  v_slot(patch, c), h * rd + i));
                    } else {
                        rotate_bf16_pairs(sr + h * rd, dr + h * rd, rd, delta[c],
                                          src->rope_base, src->pair_convention);
                    }
                }
            }
        }
    }
    return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* Standalone patch (Kamera §2: the U_m V_mᵀ term on stored rows)       */
/* ------------------------------------------------------------------ */

/* For each chunk c (tokens tok_off[c] .. tok_off[c+1]-1, placed at logical
 * positions chunk_dst_pos[c] + i of request chunk_req[c]) and each layer:
 * every patched channel value becomes rnd(x + Σ_r U·V), x the stored bf16. */
int kvo_patch_apply(kvo_pool *pool, int num_chunks, const int32_t *tok_off,
                    const int32_t *chunk_req, const int32_t *chunk_dst_pos,
                    const int32_t *block_tables, int num_reqs, int max_blocks,
                    const kvo_patch *patch)
{
    if (!pool_ok(pool) || num_chunks < 0 || !patch || patch->m <= 0)
        return KVO_ERR_INVALID;
    if (tok_off[0] != 0)
        return KVO_ERR_INVALID;
    for (int c = 0; c < num_chunks; ++c) {
        if (tok_off[c + 1] < tok_off[c])
            return KVO_ERR_INVALID;
        if (chunk_req[c] < 0 || chunk_req[c] >= num_reqs)
            return KVO_ERR_RANGE;
        const int32_t *bt = block_tables + (int64_t)chunk_req[c] * max_blocks;
        for (int64_t t = tok_off[c]; t < tok_off[c + 1]; ++t)
            if (slot_of(pool, bt, max_blocks, chunk_dst_pos[c] + (t - tok_off[c])) < 0)
                return KVO_ERR_RANGE;
    }
    const int L = pool->num_layers, cd = pool->copy_dim, rw = rot_width(pool);
    for (int c = 0; c < num_chunks; ++c) {
        const int32_t *bt = block_tables + (int64_t)chunk_req[c] * max_blocks;
        for (int l = 0; l < L; ++l) {
            for (int64_t t = tok_off[c]; t < tok_off[c + 1]; ++t) {
                int64_t d = slot_of(pool, bt, max_blocks, chunk_dst_pos[c] + (t - tok_off[c]));
                uint16_t *row[2] = {copy_row(pool, l, d), rot_row(pool, l, d)};
                int width[2] = {cd, rw};
                for (int ch = 0; ch < 2; ++ch) {
                    if (!has_patch(patch, ch))
                        continue;
                    for (int col = 0; col < width[ch]; ++col)
                        row[ch][col] = kvo_round_bf16(kvo_bf16_to_f64(row[ch][col]) +
                                                      patch_term(patch, ch, l,
                                                                 u_row(patch, tok_off, c, t),
                                                                 v_slot(patch, c), col));
                }
            }
        }
    }
    return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* Leyline splice (§2.1 directive, §2.2 Δ-rotation, §2.3 re-indexing)   */
/* ------------------------------------------------------------------ */

#define KVO_AMORTIZE 0
#define KVO_FORGET 1

/* Apply one directive per sequence.  Sequence q has the block table row
 * bt[q], length seq_lens[q] and the directive (s_start[q], s_end[q], R, m)
 * where R is stub_len[q] prefilled rows taken, in order, from the stub
 * arrays (all sequences' stubs back to back):
 *   stub_copy [L][Σ stub_len][copy_dim],  stub_rot [L][Σ stub_len][rot width]
 * AMORTIZE builds the new logical sequence out of place,
 *   new[0, s_start)                 = old[0, s_start)
 *   new[s_start, s_start + |R|)     = stub rows, verbatim
 *   new[s_start + |R| + k]          = old[s_end + k] with every rot head
 *                                     turned by R(Δ),  Δ = |R| - |S|,
 * writes it back through the block table and sets seq_lens[q] += Δ.
 * FORGET moves no data and truncates: seq_lens[q] = s_start (the caller
 * re-prefills from there).  All sequences are checked before any is edited. */
int kvo_splice(kvo_pool *pool, int num_seqs, const int32_t *block_tables, int max_blocks,
               int32_t *seq_lens, const int32_t *s_start, const int32_t *s_end,
               const int32_t *stub_len, const uint16_t *stub_copy, const uint16_t *stub_rot,
               int mode)
{
    if (!pool_ok(pool) || num_seqs < 0 || (mode != KVO_AMORTIZE && mode != KVO_FORGET))
        return KVO_ERR_INVALID;
    int64_t total_stub = 0;
    for (int q = 0; q < num_seqs; ++q) {
        if (s_start[q] < 0 || s_start[q] > s_end[q] || s_end[q] > seq_lens[q] || stub_len[q] < 0)
            return KVO_ERR_INVALID;
        total_stub += stub_len[q];
        if (mode == KVO_FORGET)
            continue;
        int64_t new_len = (int64_t)seq_lens[q] + stub_len[q] - (s_end[q] - s_start[q]);
        if ((new_len + pool->block_size - 1) / pool->block_size > max_blocks)
            return KVO_ERR_CAPACITY;
        const int32_t *bt = block_tables + (int64_t)q * max_blocks;
        int64_t hi = new_len > seq_lens[q] ? new_len : seq_lens[q];
        for (int64_t p = 0; p < hi; ++p)
            if (slot_of(pool, bt, max_blocks, p) < 0)
                return KVO_ERR_RANGE;
    }
    if (mode == KVO_FORGET) {
        for (int q = 0; q < num_seqs; ++q)
            seq_lens[q] = s_start[q];
        return KVO_OK;
    }
    if (total_stub > 0 && (!stub_copy || !stub_rot))
        return KVO_ERR_INVALID;
    const int L = pool->num_layers, cd = pool->copy_dim, rd = pool->rot_d, rh = pool->rot_heads;
    const int rw = rot_width(pool);
    int64_t stub_base = 0;
    for (int q = 0; q < num_seqs; ++q) {
        const int32_t *bt = block_tables + (int64_t)q * max_blocks;
        const int64_t n_r = stub_len[q];
        const int64_t span = s_end[q] - s_start[q];
        const int64_t delta = n_r - span;
        const int64_t old_len = seq_lens[q];
        const int64_t new_len = old_len + delta;
        uint16_t *nc = malloc((size_t)(new_len > 0 ? new_len : 1) * cd * sizeof *nc);
        uint16_t *nr = malloc((size_t)(new_len > 0 ? new_len : 1) * rw * sizeof *nr);
        if (!nc || !nr) {
            free(nc);
            free(nr);
            return KVO_ERR_INVALID;
        }
        for (int l = 0; l < L; ++l) {
            for (int64_t p = 0; p < s_start[q]; ++p) {
                int64_t s = slot_of(pool, bt, max_blocks, p);
                memcpy(nc + p * cd, copy_row(pool, l, s), (size_t)cd * sizeof *nc);
                memcpy(nr + p * rw, rot_row(pool, l, s), (size_t)rw * sizeof *nr);
            }
            for (int64_t k = 0; k < n_r; ++k) {
                int64_t p = s_start[q] + k;
                const uint16_t *sc = stub_copy + ((int64_t)l * total_stub + stub_base + k) * cd;
                const uint16_t *sr = stub_rot + ((int64_t)l * total_stub + stub_base + k) * rw;
                memcpy(nc + p * cd, sc, (size_t)cd * sizeof *nc);
                memcpy(nr + p * rw, sr, (size_t)rw * sizeof *nr);
            }
            for (int64_t k = 0; k < old_len - s_end[q]; ++k) {
                int64_t p = s_start[q] + n_r + k;
                int64_t s = slot_of(pool, bt, max_blocks, s_end[q] + k);
                memcpy(nc + p * cd, copy_row(pool, l, s), (size_t)cd * sizeof *nc);
                const uint16_t *sr = rot_row(pool, l, s);
                for (int h = 0; h < rh; ++h)
                    rotate_bf16_pairs(sr + h * rd, nr + p * rw + h * rd, rd, delta,
                                      pool->rope_base, pool->pair_convention);
            }
            for (int64_t p = 0; p < new_len; ++p) {
                int64_t s = slot_of(pool, bt, max_blocks, p);
                memcpy(copy_row(pool, l, s), nc + p * cd, (size_t)cd * sizeof *nc);
                memcpy(rot_row(pool, l, s), nr + p * rw, (size_t)rw * sizeof *nr);
            }
        }
        free(nc);
        free(nr);
        seq_lens[q] = (int32_t)new_len;
        stub_base += n_r;
    }
    return KVO_OK;
}

/* Several directives per sequence, composed (the multi-directive reading of
 * Leyline §2.2-§2.3 with the closure R(a)R(b) = R(a+b)).  Sequence q receives
 * num_dirs directives in order; directive i is given in the indexing that
 * directives 0..i-1 produced, exactly as num_dirs successive kvo_splice calls
 * would take it:
 *   (s_start[i*num_seqs + q], s_end[i*num_seqs + q], stub_len[i*num_seqs + q]).
 * Stub rows are stored directive by directive and, within a directive,
 * sequence by sequence -- the stub arrays of the successive calls back to
 * back: stub_copy [L][Σ stub_len][copy_dim], stub_rot [L][Σ stub_len][rot width].
 * Instead of rounding to bf16 after every directive, the directives are
 * applied to the ORIGIN of every logical row (an original row at position
 * p0, or a stub row that directive i wrote at position p0); the final row at
 * position p is then formed once from its origin, every rot head turned by
 * R(p - p0), and rounded once.  Only the final length is checked against the
 * block table's capacity (intermediate states are never stored). */
typedef struct {
    int64_t src;     /* >= 0: original position; < 0: stub row -1 - src */
    int64_t written; /* position the row held when it was last rounded   */
} kvo_origin;

int kvo_splice_composed(kvo_pool *pool, int num_seqs, int num_dirs, const int32_t *block_tables,
                        int max_blocks, int32_t *seq_lens, const int32_t *s_start,
                        const int32_t *s_end, const int32_t *stub_len, const uint16_t *stub_copy,
                        const uint16_t *stub_rot)
{
    if (!pool_ok(pool) || num_seqs < 0 || num_dirs < 0)
        return KVO_ERR_INVALID;
    int64_t total_stub = 0;
    for (int q = 0; q < num_seqs; ++q) {
        int64_t len = seq_lens[q];
        if (len < 0)
            return KVO_ERR_INVALID;
        for (int i = 0; i < num_dirs; ++i) {
            const int64_t a = s_start[(int64_t)i * num_seqs + q];
            const int64_t b = s_end[(int64_t)i * num_seqs + q];
            const int64_t nr = stub_len[(int64_t)i * num_seqs + q];
            if (a < 0 || a > b || b > len || nr < 0)
                return KVO_ERR_INVALID;
            len += nr - (b - a);
            total_stub += nr;
        }
        if (len > INT32_MAX)
            return KVO_ERR_INVALID;
        if ((len + pool->block_size - 1) / pool->block_size > max_blocks)
            return KVO_ERR_CAPACITY;
        const int32_t *bt = block_tables + (int64_t)q * max_blocks;
        const int64_t hi = len > seq_lens[q] ? len : seq_lens[q];
        for (int64_t p = 0; p < hi; ++p)
            if (slot_of(pool, bt, max_blocks, p) < 0)
                return KVO_ERR_RANGE;
    }
    if (total_stub > 0 && (!stub_copy || !stub_rot))
        return KVO_ERR_INVALID;
    const int L = pool->num_layers, cd = pool->copy_dim, rd = pool->rot_d, rh = pool->rot_heads;
    const int rw = rot_width(pool);
    for (int q = 0; q < num_seqs; ++q) {
        /* the origins of the logical rows, directive by directive */
        int64_t len = seq_lens[q], cap = len;
        for (int i = 0; i < num_dirs; ++i)
            cap += stub_len[(int64_t)i * num_seqs + q];
        kvo_origin *cur = malloc((size_t)(cap > 0 ? cap : 1) * sizeof *cur);
        kvo_origin *nxt = malloc((size_t)(cap > 0 ? cap : 1) * sizeof *nxt);
        if (!cur || !nxt) {
            free(cur);
            free(nxt);
            return KVO_ERR_INVALID;
        }
        for (int64_t p = 0; p < len; ++p) {
            cur[p].src = p;
            cur[p].written = p;
        }
        for (int i = 0; i < num_dirs; ++i) {
            const int64_t a = s_start[(int64_t)i * num_seqs + q];
            const int64_t b = s_end[(int64_t)i * num_seqs + q];
            const int64_t nr = stub_len[(int64_t)i * num_seqs + q];
            /* first stub row of (directive i, sequence q) */
            int64_t base = 0;
            for (int i2 = 0; i2 < num_dirs; ++i2)
                for (int q2 = 0; q2 < num_seqs; ++q2)
                    if (i2 < i || (i2 == i && q2 < q))
                        base += stub_len[(int64_t)i2 * num_seqs + q2];
            int64_t n = 0;
            for (int64_t p = 0; p < a; ++p)
                nxt[n++] = cur[p];
            for (int64_t k = 0; k < nr; ++k) {
                nxt[n].src = -1 - (base + k);
                nxt[n].written = a + k;
                ++n;
            }
            for (int64_t p = b; p < len; ++p)
                nxt[n++] = cur[p];
            kvo_origin *t = cur;
            cur = nxt;
            nxt = t;
            len = n;
        }
        const int32_t *bt = block_tables + (int64_t)q * max_blocks;
        uint16_t *nc = malloc((size_t)(len > 0 ? len : 1) * cd * sizeof *nc);
        uint16_t *nrr = malloc((size_t)(len > 0 ? len : 1) * rw * sizeof *nrr);
        if (!nc || !nrr) {
            free(cur);
            free(nxt);
            free(nc);
            free(nrr);
            return KVO_ERR_INVALID;
        }
        for (int l = 0; l < L; ++l) {
            for (int64_t p = 0; p < len; ++p) {
                const uint16_t *sc, *sr;
                if (cur[p].src >= 0) {
                    const int64_t s = slot_of(pool, bt, max_blocks, cur[p].src);
                    sc = copy_row(pool, l, s);
                    sr = rot_row(pool, l, s);
                } else {
                    const int64_t row = -1 - cur[p].src;
                    sc = stub_copy + ((int64_t)l * total_stub + row) * cd;
                    sr = stub_rot + ((int64_t)l * total_stub + row) * rw;
                }
                memcpy(nc + p * cd, sc, (size_t)cd * sizeof *nc);
                for (int h = 0; h < rh; ++h)
                    rotate_bf16_pairs(sr + h * rd, nrr + p * rw + h * rd, rd, p - cur[p].written,
                                      pool->rope_base, pool->pair_convention);
            }
            for (int64_t p = 0; p < len; ++p) {
                const int64_t s = slot_of(pool, bt, max_blocks, p);
                memcpy(copy_row(pool, l, s), nc + p * cd, (size_t)cd * sizeof *nc);
                memcpy(rot_row(pool, l, s), nrr + p * rw, (size_t)rw * sizeof *nrr);
            }
        }
        free(cur);
        free(nxt);
        free(nc);
        free(nrr);
        seq_lens[q] = (int32_t)len;
    }
    return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* Content-defined chunking of token streams                           */
/* ------------------------------------------------------------------ */
/*
 * Irminsul §2.2 ("content hash keying with CDC"): the registry is keyed by
 * content.  A Gear rolling hash over windows of 64 tokens ends a chunk
 * where the hash falls below a threshold, so chunk boundaries follow the
 * content and not its offset; each chunk is named by its xxHash64
 * fingerprint.  The fixed-window fallback (S1) fingerprints windows of 128
 * tokens instead.  The pages fix neither the Gear table nor the threshold.
 * Readings used here and nowhere else:
 *   - the Gear value of token id x is output number x (from 0) of the
 *     SplitMix64 generator (Steele, Lea and Flood, OOPSLA 2014) seeded with
 *     gear_seed: the generator's state after x + 1 steps of the golden-ratio
 *     increment, passed through its finalising mix;
 *   - h(-1) = 0 at the start of every stream and h(i) = 2 h(i-1) + G(x_i)
 *     modulo 2^64, so h(i) holds the last 64 tokens (older ones are shifted
 *     out) -- the 64-token window;
 *   - a chunk ends after token i when h(i) < threshold, and at the end of
 *     its stream; an empty stream has no chunk;
 *   - a chunk's fingerprint is XXH64 (Collet's published algorithm) of its
 *     token ids as 4-byte little-endian words, seeded with fp_seed.
 */

static uint64_t rotl64(uint64_t v, int r) { return (v << r) | (v >> (64 - r)); }

/* output number n (from 0) of SplitMix64 seeded with `seed` */
uint64_t kvo_splitmix64_at(uint64_t seed, uint64_t n)
{
    uint64_t z = seed + (n + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The five primes of XXH64. */
#define XXP1 0x9E3779B185EBCA87ull
#define XXP2 0xC2B2AE3D27D4EB4Full
#define XXP3 0x165667B19E3779F9ull
#define XXP4 0x85EBCA77C2B2AE63ull
#define XXP5 0x27D4EB2F165667C5ull

static uint64_t le64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i)
        v = (v << 8) | p[i];
    return v;
}

static uint32_t le32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

/* one accumulator step: fold an 8-byte lane into acc */
static uint64_t xx_round(uint64_t acc, uint64_t lane)
{
    acc += lane * XXP2;
    acc = rotl64(acc, 31);
    return acc * XXP1;
}

static uint64_t xx_merge(uint64_t acc, uint64_t v)
{
    acc ^= xx_round(0, v);
    return acc * XXP1 + XXP4;
}

/* XXH64 of `len` bytes: 32-byte stripes into four accumulators, then the
 * remaining 8-, 4- and 1-byte pieces, then the final avalanche. */
uint64_t kvo_xxh64(const void *data, int64_t len, uint64_t seed)
{
    const uint8_t *p = (const uint8_t *)data;
    const uint8_t *end = p + len;
    uint64_t acc;
    if (len >= 32) {
        uint64_t v1 = seed + XXP1 + XXP2, v2 = seed + XXP2, v3 = seed, v4 = seed - XXP1;
        while (end - p >= 32) {
            v1 = xx_round(v1, le64(p));
            v2 = xx_round(v2, le64(p + 8));
            v3 = xx_round(v3, le64(p + 16));
            v4 = xx_round(v4, le64(p + 24));
            p += 32;
        }
        acc = rotl64(v1, 1) + rotl64(v2, 7) + rotl64(v3, 12) + rotl64(v4, 18);
        acc = xx_merge(acc, v1);
        acc = xx_merge(acc, v2);
        acc = xx_merge(acc, v3);
        acc = xx_merge(acc, v4);
    } else {
        acc = seed + XXP5;
    }
    acc += (uint64_t)len;
    while (end - p >= 8) {
        acc ^= xx_round(0, le64(p));
        acc = rotl64(acc, 27) * XXP1 + XXP4;
        p += 8;
    }
    if (end - p >= 4) {
        acc ^= (uint64_t)le32(p) * XXP1;
        acc = rotl64(acc, 23) * XXP2 + XXP3;
        p += 4;
    }
    while (p < end) {
        acc ^= (uint64_t)(*p) * XXP5;
        acc = rotl64(acc, 11) * XXP1;
        ++p;
    }
    acc ^= acc >> 33;
    acc *= XXP2;
    acc ^= acc >> 29;
    acc *= XXP3;
    acc ^= acc >> 32;
    return acc;
}

/* XXH64 of tokens[0..n) as 4-byte little-endian words */
static uint64_t tokens_xxh64(const int32_t *tokens, int64_t n, uint64_t seed)
{
    uint8_t *buf = (uint8_t *)malloc((size_t)(n > 0 ? n : 1) * 4);
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t v = (uint32_t)tokens[i];
        buf[4 * i] = (uint8_t)v;
        buf[4 * i + 1] = (uint8_t)(v >> 8);
        buf[4 * i + 2] = (uint8_t)(v >> 16);
        buf[4 * i + 3] = (uint8_t)(v >> 24);
    }
    const uint64_t h = kvo_xxh64(buf, n * 4, seed);
    free(buf);
    return h;
}

/* The Gear hash h(i) after every token of one stream. */
void kvo_gear_hashes(const int32_t *tokens, int64_t n, uint64_t gear_seed, uint64_t *h)
{
    uint64_t acc = 0;
    for (int64_t i = 0; i < n; ++i) {
        acc = 2u * acc + kvo_splitmix64_at(gear_seed, (uint64_t)(uint32_t)tokens[i]);
        h[i] = acc;
    }
}

/* Chunks of every stream: chunk_end[k] (exclusive end, a global token
 * offset) and fingerprint[k], in stream order.  Stream s is tokens
 * [stream_off[s], stream_off[s+1]).  Returns the number of chunks; when it
 * exceeds max_chunks only the first max_chunks are written.  Returns -1 on
 * malformed offsets. */
int64_t kvo_cdc(int num_streams, const int64_t *stream_off, const int32_t *tokens,
                uint64_t gear_seed, uint64_t threshold, uint64_t fp_seed, int64_t max_chunks,
                int64_t *chunk_end, uint64_t *fingerprint)
{
    if (num_streams < 0 || (num_streams > 0 && stream_off[0] != 0))
        return -1;
    int64_t count = 0;
    for (int s = 0; s < num_streams; ++s) {
        const int64_t a = stream_off[s], b = stream_off[s + 1];
        if (b < a)
            return -1;
        uint64_t acc = 0;
        int64_t start = a;
        for (int64_t i = a; i < b; ++i) {
            acc = 2u * acc + kvo_splitmix64_at(gear_seed, (uint64_t)(uint32_t)tokens[i]);
            if (acc < threshold || i == b - 1) {
                if (count < max_chunks) {
                    chunk_end[count] = i + 1;
                    fingerprint[count] = tokens_xxh64(tokens + start, i + 1 - start, fp_seed);
                }
                ++count;
                start = i + 1;
            }
        }
    }
    return count;
}

/* Fingerprints of arbitrary token ranges [start[k], end[k]) (the fixed-window
 * fallback passes consecutive 128-token windows).  Returns -1 on a bad range. */
int kvo_fingerprint(int64_t num_ranges, const int64_t *start, const int64_t *end,
                    const int32_t *tokens, uint64_t fp_seed, uint64_t *fingerprint)
{
    for (int64_t k = 0; k < num_ranges; ++k) {
        if (end[k] < start[k] || start[k] < 0)
            return -1;
        fingerprint[k] = tokens_xxh64(tokens + start[k], end[k] - start[k], fp_seed);
    }
    return 0;
}
