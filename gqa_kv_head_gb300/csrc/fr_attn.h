// fr_attn.h -- internal interface between the fr_decode_attn entry point
// (validation, planning, workspace layout) and the tensor-core kernel.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fr_common.cuh"

namespace fr {
namespace tc {

constexpr int kMaxClusters = 24;         // clusters per 128-row tile (workspace bound)
constexpr int kMaxMergeSplits = 160;     // splits (over all row tiles) in merge-kernel mode
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a wait gives up after ~2 s

struct TcArgs {
    const __half* q16;        // f16 Q rows [M][hd] (given, or qkv_post's output)
    float* out;
    float* part_o;            // [row_tiles][n_clusters][128][hd]  (merge-kernel mode: [row_tiles][splits][128][hd])
    float2* part_ml;          // [row_tiles][n_clusters][128]      (merge-kernel mode: [row_tiles][splits][128])
    unsigned* tickets;        // [row_tiles][C]
    unsigned* status;
    int has_mask;
    int n_tok, n_head, M, n_kv;
    int n_tiles;              // KV tiles of tile_keys(...) keys
    int tiles_per_split;
    int n_clusters;           // clusters per row tile
    int C;                    // CTAs per cluster (splits per cluster)
    int merge_kernel;         // 1: write every split's state for attn_merge_kernel (C == 1)
    int early_dep;            // 1: the grid is one wave; a dependent launch may start after set-up
    int splits;               // splits per row tile
    float kq_log2;
    uint64_t wait_limit_ns;
    uint32_t probe_iters;
};

struct TcLaunch {
    TcArgs args;
    bool pdl;                 // launched right after the qkv_post grid that writes q16
    const void* k;
    const void* v;
    const void* mask;
    int64_t k_rs, v_rs, m_rs;
    int row_tiles, splits;
    int bn;                   // keys per KV tile (tile_keys)
};

int tile_keys(int hd, int n_kv, int row_tiles, int num_sms);
// 2-D f16 tensor map [rows][inner] (row stride in elements), 128-byte swizzle
// or none.
bool encode_f16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                   uint32_t box_inner, uint32_t box_rows, bool swizzle128);
fr_status launch_tc(const TcLaunch& L, int hd, cudaStream_t stream);
// Merge of the split states written in merge-kernel mode (programmatic
// dependent launch after the attention grid). ws = the workspace start, where
// the FR_TRACE build stamps its timeline (unused otherwise).
fr_status launch_merge(const float* part_o, const float2* part_ml, float* out, int M, int splits, int hd,
                       int rstride, unsigned* ws, cudaStream_t stream);

}  // namespace tc

// The kernel with the KV tile on the MMA's M side, for M <= 64 query rows
// (fr_attn_sw.cu): one KV split per CTA.
namespace sw {

constexpr int kMaxRows = 128;            // M over all slices
constexpr int kMaxSliceRows = 64;        // NQ, the MMA's N

struct SwArgs {
    float* out;
    float* part_o;            // [splits][rstride][hd] unnormalised O rows (splits > 1)
    float2* part_ml;          // [splits][rstride] (row max in log2 units, row sum)
    unsigned* status;
    const float* q;           // f32 Q rows when the kernel ropes them itself (rope_in_kernel)
    int64_t q_tok_stride;
    const int32_t* pos;
    int rope_in_kernel;       // 1: build the f16 Q tile from q/pos (qkv_post's arithmetic); 0: load q16
    int has_mask;
    int n_tok, n_head, M, n_kv;
    int keys_per_split;       // a multiple of 16; split s reads keys [s*kps, min(n_kv, (s+1)*kps))
    int splits;               // KV splits (states per row)
    int slices;               // row slices per split: CTA b takes split b / slices, rows [(b % slices)*NQ, +NQ)
    int rstride;              // rows per split block of part_o / part_ml (= M)
    unsigned* barrier;        // [2]: arrival and departure counts (grid barrier before the merge)
    int early_dep;            // 1: the grid is one wave; a dependent launch may start after set-up
    float kq_log2;
    uint64_t wait_limit_ns;
    uint32_t probe_iters;
};

struct SwMaps {
    CUtensorMap k, v, mask, q16;
};

struct SwLaunch {
    SwArgs args;
    RopeTable tb;             // rope_in_kernel only
    bool pdl;                 // programmatic dependent launch (the kernel waits before reading inputs)
    const void* q16;
    const void* k;
    const void* v;
    const void* mask;
    int64_t k_rs, v_rs, m_rs;
};

// N of the MMA (query rows padded to 16, 32 or 64) for a slice of M rows.
int rows_n(int M);
// nq: rows per slice (16, 32 or 64); the grid is args.splits * args.slices.
fr_status launch_sw(const SwLaunch& L, int hd, int nq, cudaStream_t stream);

}  // namespace sw

// Smallest workspace fr_decode_attn accepts for this shape (0 if unsupported);
// fr_decode_attn_workspace_size may ask for more so that faster plans fit.
size_t decode_attn_min_workspace_bytes(int n_tok, int n_head, int hd, int n_kv);
}  // namespace fr
