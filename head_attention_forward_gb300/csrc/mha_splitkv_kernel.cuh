// mha_splitkv_kernel.cuh - split-KV ("flash decoding") attention forward
// for a few queries against a long key/value sequence, sm_103a.
//
// What it computes: the same attention rows as the fused kernel, for Nq
// queries (the last Nq positions of the sequence) against Nk keys.  The key
// axis is cut into splits, one CTA per (batch*head, split); each CTA runs the
// online softmax of the Triton-learning blog (Puzzle 8 merge of running max
// and sum, Puzzle 9 output rescale) over its keys and emits a partial output
// normalised by its own sum plus that split's log-sum-exp.  A second kernel
// merges the splits: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
// The split of keys across workers followed by a reduction of partial results
// is the flash-decoding scheme the ML-Triton paper cites in section 3.2.
//
// With Nq <= 16 this is a memory-bound pass over K and V (about 2 d bytes
// read per multiply-add), so it runs on the CUDA cores, not the tensor
// cores: K/V tiles of 64 keys stream through a 3-slot TMA ring (128-byte
// swizzle, which also keeps the shared-memory reads below free of bank
// conflicts), two CTAs per SM keep enough bytes in flight.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "mha_wait.cuh"
#include "sm103_ptx.cuh"

namespace mha {

constexpr int kSplitMaxQ = 16;  // queries per call (decode-sized blocks)

struct SplitParams {
  const __nv_bfloat16* q;  // [BH, Nq, D]
  // paged K/V cache (used when the kernel is instantiated with PAGED):
  // logical key position t of batch entry b lives in physical block
  // block_table[b * max_blocks + t / page_size], row t % page_size
  const int* block_table;  // [B, max_blocks]
  const int* seq_lens;     // [B] keys cached per batch entry
  int page_size, max_blocks, num_heads, num_blocks;
  float* o_part;           // [BH, splits, Nq, D]  (normalised by the split's own sum)
  float* lse_part;         // [BH, splits, Nq]     (natural log; -inf when empty)
  unsigned* status;        // device status word
  long long wait_limit;
  int Nq, Nk, num_splits, tiles_per_split;
  float scale_log2;        // scale * log2(e)
  int causal;              // bottom-right aligned: query i sees keys < Nk - Nq + i + 1
};

// D: head dimension; QB: query bucket (the kernel handles Nq <= QB queries,
// QB in {1, 2, 4, 8, 16}, so a single-query decode does no work for 16).
template <int D, int QB>
struct SplitCfg {
  static constexpr int kThreads = 128;
  static constexpr int kTileKeys = 64;
  static constexpr int kStages = 3;
  static constexpr int kHalfBytes = kTileKeys * 128;  // 64 rows x 128 bytes (one swizzle atom column)
  static constexpr int kTileBytes = (D / 64) * kHalfBytes;
  static constexpr int kOffRing = 0;  // [stage][K tile, V tile]
  static constexpr int kOffQ = kStages * 2 * kTileBytes;
  static constexpr int kOffScore = kOffQ + QB * D * 4;
  static constexpr int kOffStats = kOffScore + QB * kTileKeys * 4;  // alpha, m, l
  static constexpr int kOffBar = (kOffStats + 3 * QB * 4 + 15) & ~15;  // mbarriers: 8-byte aligned
  static constexpr int kOffAbort = kOffBar + 8 * kStages;
  static_assert(kOffBar % 8 == 0 && kOffQ % 16 == 0 && kOffScore % 16 == 0, "alignment");
  static constexpr int kSmemBytes = kOffAbort + 16 + 1024;
  // output column pairs per thread group and key groups in the P V step
  static constexpr int kPairs = D / 2;
  static constexpr int kKeyGroups = kThreads / kPairs;
  static constexpr int kKeysPerGroup = kTileKeys / kKeyGroups;
  static_assert(kKeyGroups * QB * D * 4 <= kStages * 2 * kTileBytes,
                "key-group combine buffer reuses the ring");
  static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
};

// Byte offset of element (row, col) of a [rows x 64] bf16 box written by TMA
// with the 128-byte swizzle: 16-byte chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int chunk = col >> 3;
  return static_cast<uint32_t>(row * 128 + (((chunk ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

template <int D, int QB, bool PAGED>
__global__ void __launch_bounds__(SplitCfg<D, QB>::kThreads, 2)
    splitkv_partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const SplitParams p) {
  using C = SplitCfg<D, QB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int Nq = p.Nq;
  // keys of this (batch, head): fixed, or this batch entry's cached length
  // (clamped to what its block table row can address)
  const int Nk = PAGED ? min(p.seq_lens[bh / p.num_heads], p.max_blocks * p.page_size) : p.Nk;
  const int n_tiles_total = (Nk + C::kTileKeys - 1) / C::kTileKeys;
  const int t_begin = split * p.tiles_per_split;
  const int t_end = min(n_tiles_total, t_begin + p.tiles_per_split);
  const int n_tiles = max(0, t_end - t_begin);

  float* q_s = reinterpret_cast<float*>(smem + C::kOffQ);          // [QB][D]
  float* sc = reinterpret_cast<float*>(smem + C::kOffScore);       // [QB][64]
  float* alpha_s = reinterpret_cast<float*>(smem + C::kOffStats);  // [QB]
  float* m_s = alpha_s + QB;
  float* l_s = m_s + QB;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  auto full = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  auto k_tile = [&](int i) -> uint32_t { return sbase + C::kOffRing + (2 * i) * C::kTileBytes; };
  auto v_tile = [&](int i) -> uint32_t { return sbase + C::kOffRing + (2 * i + 1) * C::kTileBytes; };
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit};

  auto issue_tile = [&](int t) {  // warp 0, all lanes
    const int slot = t % C::kStages;
    if (lane == 0) ptx::mbar_arrive_expect_tx(full(slot), 2 * C::kTileBytes);
    __syncwarp();
    const int y = (t_begin + t) * C::kTileKeys;
    if constexpr (PAGED) {
      // the tile's 64 keys come from one page (pages >= 64 keys) or from
      // 64 / page_size consecutive pages, lane r loading box r (so the
      // table reads overlap); each box lands 1024-byte aligned, so the
      // 128-byte swizzle of the whole tile stays as one box's
      const int rows = min(p.page_size, C::kTileKeys);
      if (lane < C::kTileKeys / rows) {
        const int b = bh / p.num_heads, head = bh % p.num_heads;
        const int r0 = lane * rows;
        const int pos = y + r0;
        // pages past the entry's length: a block id past the cache reads as
        // zeros (pos < Nk also keeps the table read inside its row)
        const int blk = pos < Nk ? p.block_table[static_cast<size_t>(b) * p.max_blocks + pos / p.page_size]
                                 : p.num_blocks;
        const int row = pos % p.page_size;
        for (int h = 0; h < D / 64; ++h) {
          ptx::tma_load_4d(k_tile(slot) + h * C::kHalfBytes + r0 * 128, &tmK, full(slot), h * 64, row, head, blk);
          ptx::tma_load_4d(v_tile(slot) + h * C::kHalfBytes + r0 * 128, &tmV, full(slot), h * 64, row, head, blk);
        }
      }
    } else if (lane == 0) {
      for (int h = 0; h < D / 64; ++h) {
        ptx::tma_load_3d(k_tile(slot) + h * C::kHalfBytes, &tmK, full(slot), h * 64, y, bh);
        ptx::tma_load_3d(v_tile(slot) + h * C::kHalfBytes, &tmV, full(slot), h * 64, y, bh);
      }
    }
    __syncwarp();
  };

  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) ptx::mbar_init(full(i), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
  }
  // queries (fp32) and running statistics
  for (int i = tid; i < QB * D; i += C::kThreads) {
    const int qi = i / D, c = i % D;
    q_s[i] = qi < Nq ? __bfloat162float(p.q[(static_cast<size_t>(bh) * Nq + qi) * D + c]) : 0.f;
  }
  __syncthreads();
  if (warp == 0)
    for (int t = 0; t < min(n_tiles, C::kStages); ++t) issue_tile(t);

  // per-warp running statistics of queries w, w+4, w+8, w+12
  constexpr int kQPW = (QB + 3) / 4;  // queries per warp in the softmax step
  float m_run[kQPW], l_run[kQPW];
#pragma unroll
  for (int i = 0; i < kQPW; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
  }
  // P V accumulators: queries x this thread's output column pair
  const int cp = tid % C::kPairs, kg = tid / C::kPairs;
  float2 acc[QB];
#pragma unroll
  for (int i = 0; i < QB; ++i) acc[i] = make_float2(0.f, 0.f);

  int issued = min(n_tiles, C::kStages);
  bool ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int slot = t % C::kStages;
    if (!wait_one(full(slot), (t / C::kStages) & 1, ctl, kSiteMmaKV)) ok = false;
    __syncthreads();  // every thread leaves together on failure
    if (!ok || *abort_flag) {
      ok = false;
      break;
    }
    const int key0 = (t_begin + t) * C::kTileKeys;
    const uint8_t* kt = smem + (k_tile(slot) - sbase);
    const uint8_t* vt = smem + (v_tile(slot) - sbase);
    if constexpr (PAGED) {
      // V rows past the entry's length that came from its last, partly
      // filled page hold whatever the cache holds there, possibly NaN, and
      // a zero weight times NaN is NaN: clear them (the scores of those keys
      // are masked by a select, so K needs no clearing).  The clear is
      // ordered before the P V step by the barrier after the scores.
      const int valid = Nk - key0;
      if (valid < C::kTileKeys && valid % min(p.page_size, C::kTileKeys) != 0) {
        const int n16 = (C::kTileKeys - valid) * 8;  // 16-byte pieces per half
        uint8_t* vz = smem + (v_tile(slot) - sbase);
        for (int i = tid; i < (D / 64) * n16; i += C::kThreads) {
          const int h = i / n16, r = i - h * n16;
          *reinterpret_cast<uint4*>(vz + h * C::kHalfBytes + valid * 128 + r * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
      }
    }
    // ---- scores: two threads per key, each over half of d ----
    {
      const int kk = tid >> 1, half = tid & 1;
      float dot[QB];
#pragma unroll
      for (int i = 0; i < QB; ++i) dot[i] = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < D / 16; ++c8) {
        // the second half walks its chunks rotated by 4 so that the two
        // threads of a key never hit the same bank group (d = 128 puts the
        // halves in separate swizzle atoms at the same chunk positions)
        const int col = half * (D / 2) + ((c8 + 4 * half) % (D / 16)) * 8;
        const uint4 kv = *reinterpret_cast<const uint4*>(kt + (col >> 6) * C::kHalfBytes +
                                                         sw128_offset(kk, col & 63));
        const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
        float kf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(k2[e]);
          kf[2 * e] = f.x;
          kf[2 * e + 1] = f.y;
        }
#pragma unroll
        for (int qi = 0; qi < QB; ++qi) {
          if (qi < Nq) {
            const float4 qa = *reinterpret_cast<const float4*>(q_s + qi * D + col);
            const float4 qb = *reinterpret_cast<const float4*>(q_s + qi * D + col + 4);
            float t = dot[qi];
            t = fmaf(qa.x, kf[0], t); t = fmaf(qa.y, kf[1], t);
            t = fmaf(qa.z, kf[2], t); t = fmaf(qa.w, kf[3], t);
            t = fmaf(qb.x, kf[4], t); t = fmaf(qb.y, kf[5], t);
            t = fmaf(qb.z, kf[6], t); t = fmaf(qb.w, kf[7], t);
            dot[qi] = t;
          }
        }
      }
      const int kabs = key0 + kk;
#pragma unroll
      for (int qi = 0; qi < QB; ++qi) {
        const float full_dot = dot[qi] + __shfl_xor_sync(0xffffffffu, dot[qi], 1);
        if (qi < Nq && half == 0) {
          const bool visible = kabs < Nk && (!p.causal || kabs < Nk - Nq + qi + 1);
          sc[qi * C::kTileKeys + kk] = visible ? full_dot * p.scale_log2 : -INFINITY;
        }
      }
    }
    __syncthreads();
    // ---- online softmax: warp w owns queries w, w+4, w+8, w+12 ----
#pragma unroll
    for (int i = 0; i < kQPW; ++i) {
      const int qi = warp + 4 * i;
      if (qi < Nq) {
        const float x0 = sc[qi * C::kTileKeys + lane], x1 = sc[qi * C::kTileKeys + lane + 32];
        float mt = fmaxf(x0, x1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float m_new = fmaxf(m_run[i], mt);
        float a = 1.f, p0 = 0.f, p1 = 0.f;
        if (m_new != -INFINITY) {
          a = (m_run[i] == -INFINITY) ? 0.f : ptx::ex2(m_run[i] - m_new);
          p0 = ptx::ex2(x0 - m_new);
          p1 = ptx::ex2(x1 - m_new);
        }
        float ls = p0 + p1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
        l_run[i] = l_run[i] * a + ls;
        m_run[i] = m_new;
        sc[qi * C::kTileKeys + lane] = p0;
        sc[qi * C::kTileKeys + lane + 32] = p1;
        if (lane == 0) alpha_s[qi] = a;
      }
    }
    __syncthreads();
    // ---- O += P V: thread = (output column pair, key group) ----
    {
#pragma unroll
      for (int qi = 0; qi < QB; ++qi)
        if (qi < Nq) {
          const float a = alpha_s[qi];
          acc[qi].x *= a;
          acc[qi].y *= a;
        }
      const int col = 2 * cp;
#pragma unroll 4
      for (int e = 0; e < C::kKeysPerGroup; ++e) {
        const int kk = kg * C::kKeysPerGroup + e;
        const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(
            vt + (col >> 6) * C::kHalfBytes + sw128_offset(kk, col & 63));
        const float2 vf = __bfloat1622float2(v2);
#pragma unroll
        for (int qi = 0; qi < QB; ++qi)
          if (qi < Nq) {
            const float pr = sc[qi * C::kTileKeys + kk];
            acc[qi].x = fmaf(pr, vf.x, acc[qi].x);
            acc[qi].y = fmaf(pr, vf.y, acc[qi].y);
          }
      }
    }
    __syncthreads();  // the slot is free again
    if (warp == 0 && issued < n_tiles) {
      issue_tile(issued);
      ++issued;
    }
  }
  if (tid == 0 && !ok) {
    // let copies already issued land before the CTA goes away
    for (int u = max(0, issued - C::kStages); u < issued; ++u)
      drain_wait(full(u % C::kStages), (u / C::kStages) & 1, ctl);
  }
  __syncthreads();
  if (!ok) return;

  // ---- combine the key groups and write this split's partial result ----
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kQPW; ++i) {
      const int qi = warp + 4 * i;
      if (qi < Nq) {
        m_s[qi] = m_run[i];
        l_s[qi] = l_run[i];
      }
    }
  }
  float* comb = reinterpret_cast<float*>(smem + C::kOffRing);  // [groups][QB][D]
#pragma unroll
  for (int qi = 0; qi < QB; ++qi)
    if (qi < Nq) *reinterpret_cast<float2*>(comb + (kg * QB + qi) * D + 2 * cp) = acc[qi];
  __syncthreads();
  const size_t part = static_cast<size_t>(bh) * p.num_splits + split;
  for (int i = tid; i < Nq * D; i += C::kThreads) {
    const int qi = i / D, c = i % D;
    float o = 0.f;
#pragma unroll
    for (int g = 0; g < C::kKeyGroups; ++g) o += comb[(g * QB + qi) * D + c];
    const float l = l_s[qi];
    p.o_part[(part * Nq + qi) * D + c] = l > 0.f ? o / l : 0.f;
  }
  for (int qi = tid; qi < Nq; qi += C::kThreads) {
    const float l = l_s[qi];
    p.lse_part[part * Nq + qi] =
        l > 0.f ? (m_s[qi] + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }
}

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
