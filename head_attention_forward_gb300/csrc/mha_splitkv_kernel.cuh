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

#include "sm103_ptx.cuh"

namespace mha {

constexpr int kSplitMaxQ = 16;  // queries per call (decode-sized blocks)

// Merge of the split partials: one block per (query, batch*head), one thread
// per output column.  The splits' LSEs are read in parallel (thread t takes
// splits t, t + D, ...) and their weights staged in shared memory D at a
// time, so the partial outputs' loads are independent and many are in
// flight at once: a serial walk over the splits is one L2 round trip per
// split.  Up to 32 partials, the partial outputs are loaded together with
// the LSEs, before the weights are known.
template <int D>
__global__ void __launch_bounds__(D) splitkv_merge_kernel(const float* o_part, const float* lse_part,
                                                         __nv_bfloat16* o, float* lse, int Nq,
                                                         int num_splits, int parts_per_split,
                                                         const int* seq_lens, int num_heads,
                                                         long long split_keys, int max_keys) {
  static_assert(D % 32 == 0, "whole warps");
  __shared__ float red[D / 32];
  __shared__ float w_s[D];
  const int qi = blockIdx.x, bh = blockIdx.y, c = threadIdx.x;
  const int lane = c & 31, warp = c >> 5;
  const size_t base = static_cast<size_t>(bh) * num_splits;
  // num_splits partials per head, parts_per_split of them per key split.
  // Paged caches: an entry has only the partials of the splits that hold
  // some of its keys (the partial pass skips the others and leaves their
  // slots unwritten).
  // launched as a programmatic dependent of the partial pass: its CTAs may
  // be resident before that pass ends, so wait for its results here
  ptx::griddep_wait();
  int ns = num_splits;
  if (seq_lens) {
    const long long nk = max(0, min(seq_lens[bh / num_heads], max_keys));
    ns = static_cast<int>(min(static_cast<long long>(num_splits),
                              parts_per_split * ((nk + split_keys - 1) / split_keys)));
  }
  auto lse_of = [&](int s) { return lse_part[(base + s) * Nq + qi]; };
  const float* src = o_part + (base * Nq + qi) * D + c;
  const size_t stride = static_cast<size_t>(Nq) * D;
  // Up to kMergeRegs partials (the usual case): every load, the LSEs and
  // this thread's column of each partial output, is issued before the first
  // result is used, so the merge costs one round trip to L2, not three.
  constexpr int kMergeRegs = 32;
  const bool in_regs = ns <= kMergeRegs;
  float ov[kMergeRegs];
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kMergeRegs; ++i) ov[i] = i < ns ? src[i * stride] : 0.f;
  }
  // the largest split LSE
  const float my_lse = c < ns ? lse_of(c) : -INFINITY;
  float m = my_lse;
  for (int s = c + D; s < ns; s += D) m = fmaxf(m, lse_of(s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float lmax = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) lmax = fmaxf(lmax, red[w]);
  float out = 0.f, lse_row = -INFINITY;
  if (lmax != -INFINITY) {  // uniform across the block
    float wsum = 0.f, acc = 0.f;
    if (in_regs) {
      if (c < ns) w_s[c] = __expf(my_lse - lmax);
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kMergeRegs; ++i) {
        if (i < ns) {
          const float w = w_s[i];
          wsum += w;
          acc = fmaf(w, ov[i], acc);
        }
      }
    } else {
      for (int s0 = 0; s0 < ns; s0 += D) {
        const int n = min(D, ns - s0);
        __syncthreads();  // the previous chunk's weights are no longer read
        if (c < n) w_s[c] = __expf((s0 == 0 ? my_lse : lse_of(s0 + c)) - lmax);
        __syncthreads();
#pragma unroll 8
        for (int i = 0; i < n; ++i) {
          const float w = w_s[i];
          wsum += w;
          acc = fmaf(w, src[(s0 + i) * stride], acc);
        }
      }
    }
    out = acc / wsum;
    lse_row = lmax + __logf(wsum);
  }
  o[(static_cast<size_t>(bh) * Nq + qi) * D + c] = __float2bfloat16_rn(out);
  if (c == 0) lse[static_cast<size_t>(bh) * Nq + qi] = lse_row;
}

}  // namespace mha
