// mha_splitkv_kernel.cuh - the merge step of split-KV ("flash decoding")
// attention for a few queries against a long key/value sequence, sm_103a.
//
// The key axis of each head is cut into splits; the partial pass (the
// persistent attention kernel of mha_fwd_kernel.cuh in split mode) runs the
// online softmax of the Triton-learning blog (Puzzle 8 merge of running max
// and sum, Puzzle 9 output rescale) over each split's keys and emits a
// partial output normalised by the split's own sum plus that split's
// log-sum-exp.  The kernel here merges the splits:
//   LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
// The split of keys across workers followed by a reduction of partial
// results is the flash-decoding scheme the ML-Triton paper cites in section
// 3.2.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace mha {

constexpr int kSplitMaxQ = 16;  // queries per call (decode-sized blocks)

// Merge of the split partials: one block per (query, batch*head), one thread
// per output column.
template <int D>
__global__ void __launch_bounds__(D) splitkv_merge_kernel(const float* o_part, const float* lse_part,
                                                         __nv_bfloat16* o, float* lse, int Nq,
                                                         int num_splits, const int* seq_lens,
                                                         int num_heads, long long split_keys,
                                                         int max_keys) {
  const int qi = blockIdx.x, bh = blockIdx.y, c = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * num_splits;
  // paged caches: an entry has only the splits that hold some of its keys
  // (the partial pass may skip the others and leave their slots unwritten)
  int ns = num_splits;
  if (seq_lens) {
    const long long nk = max(0, min(seq_lens[bh / num_heads], max_keys));
    ns = static_cast<int>(min(static_cast<long long>(num_splits), (nk + split_keys - 1) / split_keys));
  }
  float lmax = -INFINITY;
  for (int s = 0; s < ns; ++s) lmax = fmaxf(lmax, lse_part[(base + s) * Nq + qi]);
  float out = 0.f, lse_row = -INFINITY;
  if (lmax != -INFINITY) {
    float wsum = 0.f, acc = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float w = __expf(lse_part[(base + s) * Nq + qi] - lmax);
      wsum += w;
      acc = fmaf(w, o_part[((base + s) * Nq + qi) * D + c], acc);
    }
    out = acc / wsum;
    lse_row = lmax + __logf(wsum);
  }
  o[(static_cast<size_t>(bh) * Nq + qi) * D + c] = __float2bfloat16_rn(out);
  if (c == 0) lse[static_cast<size_t>(bh) * Nq + qi] = lse_row;
}

}  // namespace mha
