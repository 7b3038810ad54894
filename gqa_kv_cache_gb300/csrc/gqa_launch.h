// Host-side entry points of the kernels, used by the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gqa_common.cuh"

namespace gqa {

// CUDA-core decode kernel (gqa_simt.cu).
bool simt_supports(int D, int G);
int simt_tile();
int simt_ctas_per_sm(bool bf16, int D, int G);  // occupancy of that instantiation
cudaError_t simt_launch(const DecodeParams &p, bool bf16, cudaStream_t st);

// TMA-ring + tensor-core decode kernel (gqa_tc.cu).
struct TcMaps {
    CUtensorMap k, v;      // tiled maps over the key / value cache, 128-byte swizzle
    CUtensorMap k16, v16;  // dense caches: the same with a box of kDenseBoxRows slots
};
// A dense cache's tile is one 64-slot box when every part of it is read; a
// tile that is only partly read (a unit's last tile, a window's first) is
// copied in boxes of kDenseBoxRows slots, those that hold a slot the step
// reads. A paged cache's box is its block (at most the tile).
constexpr int kDenseBoxRows = 16;
bool tc_supports(bool bf16, int D, int G, bool paged, int block_size);  // bf16: the cache
int tc_tile();
int tc_ctas_per_sm(bool kv8, int unit_rows);   // resident CTAs per SM of the instantiation
cudaError_t tc_launch(const DecodeParams &p, const TcMaps &maps, cudaStream_t st);
// The tcgen05 form of multi-token units of 17 to 32 query rows over a bf16
// cache (gqa_tc_multi.cu): whether it takes the step, and its launch.
bool tc5_takes(const DecodeParams &p);
cudaError_t tc5_launch_multi(const DecodeParams &p, const TcMaps &maps, cudaStream_t st);

// Small-cache kernel: one cluster of CTAs per unit, the unit staged in their
// shared memory (gqa_unit.cu). cap_rows: the row capacity in slots.
bool unit_supports(bool bf16, int D, int G, long long cap_rows);
size_t unit_smem_bytes(bool bf16, int D, int G, long long rows, int cl);
int unit_ctas_per_sm(bool bf16, int D, int G, long long cap_rows);
int unit_cluster(long long cap_rows, long long units, int sms);   // CTAs a unit
cudaError_t unit_launch(const DecodeParams &p, bool bf16, long long cap_rows, int sms, cudaStream_t st);

// Content validation (gqa_validate.cu). *d_result must be zero on entry; the
// kernel sets it to 1 on any violation. attend = 1 checks the read-only
// attend's reading of lengths (the number of valid slots).
cudaError_t validate_launch(const int32_t *lengths, const int32_t *slot_ids,
                            const int32_t *block_table, int B, int R, int Smax,
                            int num_blocks, int block_size, int max_blocks, int attend,
                            const int32_t *cu_q, int T, int32_t *d_result, cudaStream_t st);

}  // namespace gqa
