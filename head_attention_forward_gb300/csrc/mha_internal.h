// mha_internal.h - host-side helpers shared by the library's translation
// units (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>

namespace mha_host {

// Once per device: architecture check, driver entry point lookup, status
// word address.  Returns an mha_status code; on success fills dev / status.
int device_setup(int* dev, unsigned** status);

// Multiprocessor count of a device device_setup has accepted.
int device_sms(int dev);

// 3-D TMA view [BH][N][d] of a contiguous bf16 tensor, box 64 x box_rows x 1,
// 128-byte swizzle; rows past N read as zero.
bool encode_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);

// 4-D TMA view [num_blocks][H][page_size][d] of a paged bf16 K or V cache,
// box 64 x box_rows x 1 x 1 (box_rows <= page_size), 128-byte swizzle;
// out-of-range block ids read as zero.
bool encode_paged_map(CUtensorMap* map, const void* base, int num_blocks, int H, int page_size, int d,
                      int box_rows);

// The partial pass of split-KV decoding on the tensor cores (the persistent
// attention kernel in split mode): Nq <= 32 queries per head against Nk
// keys, num_splits runs of tiles_per_split 128-key tiles, fp32 partial
// outputs for the merge kernel.  tile_counter is one int of device memory
// the pass zeroes (on `st`) and then uses to hand out work tiles.
// device_setup must have accepted `dev`.
int fwd_split_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      int* tile_counter, int BH, int Nq, int Nk, int d, float scale, bool causal,
                      int num_splits, int tiles_per_split, int dev, unsigned* status, cudaStream_t st);

// The same partial pass over a paged K/V cache (the layout mha_fwd_paged
// documents): batch entry b holds min(seq_lens[b], max_blocks * page_size)
// keys; splits past an entry's keys are not computed and their partials
// are left as they were (the merge reads only the splits an entry has).
int fwd_paged_partial(const void* q, const void* k_cache, const void* v_cache,
                      const int* block_table, const int* seq_lens, float* o_part, float* lse_part,
                      int* tile_counter, int B, int H, int Nq, int d, int page_size, int num_blocks,
                      int max_blocks, float scale, bool causal, int num_splits, int tiles_per_split, int dev,
                      unsigned* status, cudaStream_t st);

// Cycle budget of every device-side wait for launches made now.
long long wait_limit();

bool aligned16(const void* p);

// True when [a, a+na) and [b, b+nb) overlap.
bool overlap(const void* a, size_t na, const void* b, size_t nb);

}  // namespace mha_host
