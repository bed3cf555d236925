// kv_launch.h -- internal launchers (one per kernel family).
#pragma once

#include "kv_internal.h"

namespace kvr {

// Row shapes with a compiled kernel.
enum class RowKind {
    Mla,  // verbatim 512 + rotary 1 x 64 (c_KV + k_pe)
    Gqa,  // verbatim 1024 + rotary 8 x 128 (V + K, 8 KV heads)
    Gqa4, // verbatim 512 + rotary 4 x 128 (V + K, 4 KV heads)
    Mha   // verbatim 4096 + rotary 32 x 128 (V + K, 32 heads)
};

cudaError_t launch_delta_table(const TableParams &p, cudaStream_t stream);
cudaError_t launch_relocate(const RelocParams &p, RowKind kind, cudaStream_t stream);
// Patched relocation / in-place patch on the tensor cores (tcgen05), ranks <= 16
// (larger ranks take launch_relocate's per-element patch).
bool patch_tc_supported(const RelocParams &p, RowKind kind);
cudaError_t launch_patch_tc(const RelocParams &p, RowKind kind, cudaStream_t stream);
int patch_tc_launches(const RelocParams &p, RowKind kind); // kernels launch_patch_tc issues
// Launches one ticketed block per tile; `blocks` = p.total_tickets.
cudaError_t launch_splice(const SpliceParams &p, RowKind kind, cudaStream_t stream);
// Composed splice: one ticketed block per tile of p.tiles.
cudaError_t launch_splice_composed(const ComposedParams &p, RowKind kind, cudaStream_t stream);
// Block-aligned splice by remapping: the data kernel, then the commit of the
// permuted block-table rows (dynamic shared memory: max_blocks entries).
cudaError_t launch_remap(const RemapParams &p, RowKind kind, cudaStream_t stream);
constexpr int32_t kMaxRemapBlocks = 48 * 1024; // block-table entries one commit block holds
cudaError_t launch_wait_check(uint32_t *flag, uint32_t *status, int64_t limit_ns,
                              cudaStream_t stream);
// Debug checks (kv_set_debug_checks): relocation overlap, duplicate blocks.
cudaError_t launch_overlap_check(const OverlapParams &p, cudaStream_t stream);
cudaError_t launch_dup_block_check(const DupBlockParams &p, cudaStream_t stream);
// Content-defined chunking: flags, scan, emit (+ fingerprint) kernels.
int64_t cdc_blocks(int64_t total_tokens);
cudaError_t launch_cdc(const CdcParams &p, cudaStream_t stream);
cudaError_t launch_fingerprint(const FingerprintParams &p, cudaStream_t stream);
constexpr int kCdcLaunches = 3;

// Rows per tile of each kind for the relocation (launch_relocate).
inline int tile_rows(RowKind kind)
{
    switch (kind) {
    case RowKind::Mla:
        return kTileMla;
    case RowKind::Gqa:
        return kTileGqa;
    case RowKind::Gqa4:
        return kTileGqa4;
    case RowKind::Mha:
        return kTileMha;
    }
    return kTileGqa;
}

// Rows per tile of the in-place passes over multi-head rows (the ticketed
// splice, the composed splice and the block-table remap): half the rows of
// the relocation's tiles, at three (splices: 288-thread blocks) or four
// (remap) blocks per SM.
constexpr int kInPlaceTileGqa = 8;
constexpr int kInPlaceTileGqa4 = 16;
constexpr int kInPlaceTileMha = 2;

// Rows per tile of launch_splice, launch_splice_composed (and the host plan
// of its tiles) and launch_remap; the kernels' G::T must equal it.
inline int inplace_tile_rows(RowKind kind)
{
    switch (kind) {
    case RowKind::Mla:
        return kTileMla;
    case RowKind::Gqa:
        return kInPlaceTileGqa;
    case RowKind::Gqa4:
        return kInPlaceTileGqa4;
    case RowKind::Mha:
        return kInPlaceTileMha;
    }
    return kInPlaceTileGqa;
}

} // namespace kvr
