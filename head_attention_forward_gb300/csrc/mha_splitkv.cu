// mha_splitkv.cu - host side of the split-KV attention forward (a few
// queries against a long key/value sequence, contiguous or paged): argument
// checks, split count, workspace layout, and the partial + merge launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "mha_fwd.h"
#include "mha_internal.h"
#include "mha_splitkv_kernel.cuh"

namespace {

using namespace mha_host;

// The partial pass (the persistent attention kernel in split mode, one CTA
// per SM) takes 128-key tiles and hands (head, split) work tiles out at run
// time.  Each work tile costs a pipeline drain at its end, so fewer, longer
// ones do better until the last ones leave CTAs idle: about six per CTA
// measured best on decode shapes (88-98% of the HBM copy rate against
// 84-88% with 32 per CTA).
//
// Small problems (at most kOneWaveTiles K/V tiles per SM) are latency-bound
// rather than bandwidth-bound: there at most one work tile per SM, with an
// even number of K/V tiles (the two stages take alternate tiles), measured
// 8-33% faster than six per SM (one query on 32 heads x 4k keys: 16.5 us
// against 20.6; 8 heads x 16k keys: 17.5 against 26.1).  That needs fewer
// heads than SMs, and a head count whose splits keep at least 4/5 of the
// SMs busy.  At ~108 tiles per SM six per SM was still 1.4% ahead.
//
// Fixed constants (the SM count of a GB300) keep the workspace size a pure
// function of the problem shape.
constexpr int kTileKeys = 128;
constexpr int kPlanSMs = 152;
constexpr int kTargetTiles = 6 * kPlanSMs;
constexpr int kOneWaveTiles = 64;

struct Plan {
  int splits = 0, tiles_per_split = 0;
  size_t o_part_bytes = 0, lse_part_bytes = 0, lse_off = 0, counter_off = 0, total = 0;
};

// Split count and workspace layout: o_part fp32 [BH, 2 * splits, Nq, d],
// then (16-byte aligned) lse_part fp32 [BH, 2 * splits, Nq], then (16-byte
// aligned) the partial pass's work-tile counter (one int in 16 bytes).  A
// split is a run of tiles_per_split 128-key tiles, and gives two partials:
// the partial pass alternates its tiles between two stages.
constexpr int kPartsPerSplit = 2;
Plan make_plan(long long BH, int Nq, int Nk, int d, int num_splits) {
  Plan pl;
  const int tiles = (Nk + kTileKeys - 1) / kTileKeys;
  const bool one_wave = num_splits == 0 && BH < kPlanSMs &&
                        BH * tiles <= static_cast<long long>(kOneWaveTiles) * kPlanSMs &&
                        5 * (kPlanSMs / BH) * BH >= 4 * kPlanSMs;
  int want = num_splits > 0 ? num_splits
             : one_wave     ? static_cast<int>(kPlanSMs / BH)
                            : static_cast<int>(std::max<long long>(1, (kTargetTiles + BH - 1) / BH));
  want = std::max(1, std::min(want, tiles));
  pl.tiles_per_split = (tiles + want - 1) / want;
  if (one_wave && pl.tiles_per_split > 1 && (pl.tiles_per_split & 1)) ++pl.tiles_per_split;
  pl.splits = (tiles + pl.tiles_per_split - 1) / pl.tiles_per_split;
  pl.o_part_bytes = static_cast<size_t>(BH) * kPartsPerSplit * pl.splits * Nq * d * 4;
  pl.lse_part_bytes = static_cast<size_t>(BH) * kPartsPerSplit * pl.splits * Nq * 4;
  pl.lse_off = (pl.o_part_bytes + 15) & ~static_cast<size_t>(15);
  pl.counter_off = (pl.lse_off + pl.lse_part_bytes + 15) & ~static_cast<size_t>(15);
  pl.total = pl.counter_off + 16;
  return pl;
}

// the split pass keeps every query row in the first softmax warp
static_assert(mha::kSplitMaxQ <= 32, "query rows per split-pass work tile");

int check_shape(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || num_splits < 0) return MHA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return MHA_ERR_UNSUPPORTED_DIM;
  if (Nq > mha::kSplitMaxQ) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffll) return MHA_ERR_INVALID_ARG;
  return MHA_OK;
}

// Paged caches: what the merge needs to count each entry's partials.
struct PagedSplits {
  const int* seq_lens = nullptr;  // null: every head has all the partials
  int num_heads = 1, max_keys = 0;
  long long split_keys = 1;       // keys per split
};

// Merge kernel: the splits' partial outputs into O (bf16) and LSE.
int launch_merge(const float* o_part, const float* lse_part, void* o, float* lse, long long BH,
                 int Nq, int d, int splits, cudaStream_t st, const PagedSplits& ps = PagedSplits()) {
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(static_cast<unsigned>(Nq), static_cast<unsigned>(BH), 1);
  mcfg.blockDim = dim3(static_cast<unsigned>(d), 1, 1);
  mcfg.stream = st;
  // programmatic dependent launch: the merge grid is set up while the
  // partial pass runs and starts on the SMs it leaves; the kernel waits for
  // the partials before reading them
  cudaLaunchAttribute attr[1] = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
  cudaError_t err;
  const int parts = kPartsPerSplit * splits;
  if (d == 64)
    err = cudaLaunchKernelEx(&mcfg, mha::splitkv_merge_kernel<64>, o_part, lse_part, ob, lse, Nq, parts,
                             kPartsPerSplit, ps.seq_lens, ps.num_heads, ps.split_keys, ps.max_keys);
  else
    err = cudaLaunchKernelEx(&mcfg, mha::splitkv_merge_kernel<128>, o_part, lse_part, ob, lse, Nq, parts,
                             kPartsPerSplit, ps.seq_lens, ps.num_heads, ps.split_keys, ps.max_keys);
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t mha_fwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_shape(B, H, Nq, Nk, d, num_splits) != MHA_OK) return 0;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || Nq == 0 || Nk == 0) return 0;
  return make_plan(BH, Nq, Nk, d, num_splits).total;
}

int mha_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Nq, int Nk, int d, float scale, int causal, int num_splits, void* workspace,
               size_t workspace_bytes, void* stream) {
  int rc = check_shape(B, H, Nq, Nk, d, num_splits);
  if (rc != MHA_OK) return rc;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MHA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || Nq == 0) return MHA_OK;
  if (Nk == 0) return MHA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !workspace) return MHA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return MHA_ERR_MISALIGNED;
  const Plan pl = make_plan(BH, Nq, Nk, d, num_splits);
  if (workspace_bytes < pl.total) return MHA_ERR_INVALID_ARG;
  if (BH * pl.splits > 0x7fffffffll) return MHA_ERR_INVALID_ARG;  // work tiles are counted in int
  const size_t qb = static_cast<size_t>(BH) * Nq * d * 2, kb = static_cast<size_t>(BH) * Nk * d * 2;
  const size_t lb = static_cast<size_t>(BH) * Nq * 4;
  // outputs and workspace must not overlap the inputs or each other
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {qb, kb, kb};
  for (int i = 0; i < 3; ++i)
    if (overlap(o, qb, ins[i], in_bytes[i]) || overlap(lse, lb, ins[i], in_bytes[i]) ||
        overlap(workspace, pl.total, ins[i], in_bytes[i]))
      return MHA_ERR_INVALID_ARG;
  if (overlap(o, qb, lse, lb) || overlap(o, qb, workspace, pl.total) ||
      overlap(lse, lb, workspace, pl.total))
    return MHA_ERR_INVALID_ARG;

  int dev = 0;
  unsigned* status = nullptr;
  rc = device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.lse_off);
  int* counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + pl.counter_off);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = fwd_split_partial(q, k, v, o_part, lse_part, counter, static_cast<int>(BH), Nq, Nk, d, scale,
                         causal != 0, pl.splits, pl.tiles_per_split, dev, status, st);
  if (rc != MHA_OK) return rc;
  return launch_merge(o_part, lse_part, o, lse, BH, Nq, d, pl.splits, st);
}

int mha_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                  const int* seq_lens, void* o, float* lse, int B, int H, int Nq, int d,
                  int page_size, int num_blocks, int max_blocks, float scale, int causal,
                  int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (max_blocks < 0 || num_blocks < 0 || page_size <= 0) return MHA_ERR_INVALID_ARG;
  if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0) return MHA_ERR_INVALID_ARG;
  const long long max_keys = static_cast<long long>(max_blocks) * page_size;
  if (max_keys > 0x7fffffffll) return MHA_ERR_INVALID_ARG;
  int rc = check_shape(B, H, Nq, static_cast<int>(max_keys), d, num_splits);
  if (rc != MHA_OK) return rc;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MHA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || Nq == 0) return MHA_OK;
  if (max_blocks == 0 || num_blocks == 0) return MHA_ERR_INVALID_ARG;
  // the kernel addresses a page as block * H + head, in int, with block up
  // to num_blocks (the id that reads as zeros)
  if ((static_cast<long long>(num_blocks) + 1) * H > 0x7fffffffll) return MHA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse || !workspace)
    return MHA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(lse) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(block_table) & 3) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3))
    return MHA_ERR_MISALIGNED;
  const Plan pl = make_plan(BH, Nq, static_cast<int>(max_keys), d, num_splits);
  if (workspace_bytes < pl.total) return MHA_ERR_INVALID_ARG;
  if (BH * pl.splits > 0x7fffffffll) return MHA_ERR_INVALID_ARG;  // work tiles are counted in int
  const size_t qb = static_cast<size_t>(BH) * Nq * d * 2;
  const size_t cb = static_cast<size_t>(num_blocks) * H * page_size * d * 2;
  const size_t lb = static_cast<size_t>(BH) * Nq * 4;
  const size_t tb = static_cast<size_t>(B) * max_blocks * 4, sb = static_cast<size_t>(B) * 4;
  const void* ins[5] = {q, k_cache, v_cache, block_table, seq_lens};
  const size_t in_bytes[5] = {qb, cb, cb, tb, sb};
  for (int i = 0; i < 5; ++i)
    if (overlap(o, qb, ins[i], in_bytes[i]) || overlap(lse, lb, ins[i], in_bytes[i]) ||
        overlap(workspace, pl.total, ins[i], in_bytes[i]))
      return MHA_ERR_INVALID_ARG;
  if (overlap(o, qb, lse, lb) || overlap(o, qb, workspace, pl.total) ||
      overlap(lse, lb, workspace, pl.total))
    return MHA_ERR_INVALID_ARG;

  int dev = 0;
  unsigned* status = nullptr;
  rc = device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.lse_off);
  int* counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + pl.counter_off);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = fwd_paged_partial(q, k_cache, v_cache, block_table, seq_lens, o_part, lse_part, counter, B, H, Nq,
                         d, page_size, num_blocks, max_blocks, scale, causal != 0, pl.splits,
                         pl.tiles_per_split, dev, status, st);
  if (rc != MHA_OK) return rc;
  PagedSplits ps;
  ps.seq_lens = seq_lens;
  ps.num_heads = H;
  ps.max_keys = static_cast<int>(max_keys);
  ps.split_keys = static_cast<long long>(pl.tiles_per_split) * kTileKeys;
  return launch_merge(o_part, lse_part, o, lse, BH, Nq, d, pl.splits, st, ps);
}

}  // extern "C"
