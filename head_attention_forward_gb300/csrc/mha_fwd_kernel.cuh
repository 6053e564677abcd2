// mha_fwd_kernel.cuh - fused attention forward for sm_103a (GB300).
//
// What it computes: the FlashAttention-2 forward pass of the ML-Triton paper
// (section 2.5, Algorithm 1): for a tile of queries, loop over key/value
// tiles, S = Q K^T, online softmax with running row max m and row sum l,
// O += P V, and one final normalisation.  The running statistics follow the
// Triton-learning blog (Puzzle 8: sum' = sum * exp(m1 - m2) + sum exp(x - m2);
// Puzzle 9: the output is rescaled by the same factor), with the division by
// l deferred to the end, and exp written as exp2 of a pre-scaled argument
// (blog, Puzzle 8: exp(x) = 2^(log2(e) x)).
//
// How it maps to GB300.  A work tile is 256 query rows of one (batch,
// head), split into two 128-row Q tiles.  The kernel is persistent: one CTA
// per SM walks its share of the work tiles, so TMEM, barriers and the K/V
// ring are set up once and the next tile's loads overlap this one's tail.
// The work tiles come in snake rounds over heads, or (HMAJOR, d = 128 with
// K/V beyond L2) head-major, causal m-blocks paired for equal cost.
//   warp 0      TMA producer for K_j / V_j of every work tile in turn, into
//               a ring of shared-memory stages guarded by full/empty
//               mbarriers (the producer/consumer tokens of the Triton
//               warp-specialisation notes: acquire -> expect bytes -> TMA
//               copy; consumer waits -> uses -> releases).
//   warp 2      TMA producer for Q0/Q1 of each work tile, as soon as the
//               tensor core no longer reads the Q buffer set it reuses.
//   warp 1      MMA issuer: S_j(s) = Q_s K_j^T with tcgen05.mma into
//               TMEM, then O(s) += P_j(s) V_j with P read straight from
//               TMEM.  The whole warp runs the issue loop (so descriptors and
//               loop state are warp-uniform) and one elected lane issues
//               each batch of MMAs and commits.  Also allocates / frees TMEM.
//   warps 4-7   softmax warpgroup for Q tile 0 (TMEM lanes 0-127, one query
//   warps 8-11  row per thread), softmax warpgroup for Q tile 1.  Each reads
//               its S row from TMEM, masks, updates m and l, writes P (bf16)
//               back over S, rescales O in TMEM when its max moved (the
//               correction stage), and finally writes O / l and the LSE
//               (at d = 128 through a shared-memory chunk and TMA stores).
//   warp 3      idle (keeps the softmax warpgroups aligned to TMEM lanes).
// The two Q tiles ping-pong: while one softmax warpgroup works on its S, the
// tensor core runs the other tile's GEMMs (the cooperative M-split of the
// warp-specialisation notes, one consumer group per half of the rows).
//
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+W), O1 [384,384+W),
// W = D, or 80 in the square pass at d = 64 (column 64 then holds the row
// sum of P, formed by the tensor core).  P_j(s) (128 keys as 64 packed
// bf16x2 columns) overwrites S(s) cols [0,64).
// The tensor pipe executes one thread's MMAs in issue order, so issuing
// S_{j+1}(s) after PV_j(s) cannot clobber P_j(s) before it is read.
//
// Split mode (SPLIT) serves split-KV decoding, a few queries against a long
// key sequence: work tiles are (head, key split) pairs that warp 0 hands out
// at run time; the queries (at most 32) sit in the first softmax warp of
// each stage and the other softmax warps have no work; a split's K/V tiles
// alternate between the stages, so the two stages' softmax warps work on
// consecutive tiles at once; each stage writes an fp32 partial output and
// its LSE for a merge kernel (two partials per split).  The split pass runs
// between two programmatic-dependent launches: after the kernel that zeroes
// its work-tile counter, before the merge kernel.  PAGED gathers each
// 128-key tile of a paged K/V cache from page-sized TMA boxes named by a
// block table (at d = 128 one box holds both d-halves of its rows).
//
// Every mbarrier wait is bounded (clock64 budget).  A wait that runs out
// records a code in the device status word, raises a CTA-wide abort flag
// that ends every other wait at once, and the CTA then drains its own
// in-flight copies and MMAs (again with a bound) and frees TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "mha_wait.cuh"
#include "sm103_ptx.cuh"

namespace mha {

struct FwdParams {
  __nv_bfloat16* o;    // [BH, N, D]
  float* lse;          // [BH, N]
  unsigned* status;    // device status word
  long long wait_limit;  // SM cycles per wait
  int N;
  int num_mblocks;     // ceil(N / 256)
  int BH;              // batch * heads; work tiles are (bh, m-block) pairs
  // split mode only: Nq <= 32 queries per head (one Q tile, rows past Nq
  // read as zeros) against Nk keys cut into num_splits runs of tiles_per_split
  // K/V tiles; work tiles are (bh, split) pairs, and each stage writes an
  // fp32 partial output for its half of the split's tiles, normalised by its
  // own sum, plus its log-sum-exp
  int Nq, Nk, num_splits, tiles_per_split;
  float* o_part;       // [BH, 2 * num_splits, Nq, D] (one partial per split and stage)
  float* lse_part;     // [BH, 2 * num_splits, Nq]
  float scale_log2;    // scale * log2(e)
  // paged mode only (split mode over a paged cache): key t of batch entry
  // b = bh / num_heads is row t % page_size of cache block
  // block_table[b * max_blocks + t / page_size]; the entry holds
  // min(seq_lens[b], max_blocks * page_size) keys and Nk is that bound
  const int* block_table;  // [B, max_blocks]
  const int* seq_lens;     // [B]
  int page_size, max_blocks, num_heads, num_blocks;
  int* tile_counter;       // split mode: work tiles handed out so far past the grid (zero at launch)
};

template <int D, bool SPLIT = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int kBlockM = 128;  // query rows per softmax warpgroup
  static constexpr int kBlockN = 128;  // keys per K/V tile
  static constexpr int kHalves = D / 64;  // 128-byte swizzle atoms across d
  static constexpr int kHalfBytes = 128 * 128;  // 128 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  // square mode at d = 64: the tensor core also sums each row's bf16 P: the
  // V operand of P V gets a 65th column of ones, read from a constant tile
  // after the ring (its descriptor's N-atom stride points there), and O(s)
  // holds that sum in column 64
  static constexpr bool kSumCol = !SPLIT && D == 64;
  static constexpr int kONcols = kSumCol ? 80 : D;  // P V's N (a multiple of 16)
  static constexpr int kStages = (D == 128) ? 4 : 8;
  // Q buffer sets: with two, the next work tile's Q loads during this one
  static constexpr int kQSets = (D == 128) ? 1 : 2;
  // square mode at d = 128: staging for the O epilogue, one 32-row chunk per
  // TMEM lane quarter, written to HBM by TMA stores; the warps of the two
  // stages on that lane quarter share it, in the order of their epilogues
  // (there is no room for a chunk per warp).  At d = 64 the softmax warps
  // store their rows directly, which measured faster there (2-4%) while the
  // staged stores gained 1-2% at d = 128.
  static constexpr int kOSets = (SPLIT || D == 64) ? 0 : 1;
  static constexpr int kOChunkBytes = 32 * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQSets * 2 * kTileBytes;
  static constexpr int kOffO = kOffKV + kStages * kTileBytes;
  // the ones tile: 128 keys x one 128-byte swizzle row, 8-key groups 1 KiB apart
  static constexpr int kOffOnes = kOffO + kOSets * 4 * kOChunkBytes;
  static constexpr int kOffBar = kOffOnes + (kSumCol ? 16 * 1024 : 0);
  // split mode: ring of work-tile ids from the K/V producer to the other
  // roles (Q producer, MMA issuer, the softmax warps that hold query rows)
  static constexpr int kTileRing = 8;
  // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_ready[2] o_full[2] drain
  // tail (paged mode: the copy of a V tile whose last rows get cleared)
  // tile_full[R] tile_empty[R] o_free[4] (a shared O staging chunk is free)
  static constexpr int kNumBars = 4 + 2 * kStages + 2 + 2 + 2 + 1 + 1 + 2 * kTileRing + 4;
  static constexpr int kOffTileIds = kOffBar + 8 * kNumBars;
  static constexpr int kOffTmemSlot = kOffTileIds + 4 * kTileRing;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kOffBar % 8 == 0 && kOffKV % 1024 == 0 && kOffO % 1024 == 0 && kOffOnes % 1024 == 0,
                "mbarrier / swizzle-atom alignment");
  static constexpr int kThreads = 384;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
  // the running max only moves (and O is only rescaled) once it has grown
  // by more than this many powers of two; P stays <= 2^8 meanwhile.
  static constexpr float kRescaleThreshold = 8.0f;
};

// The O tensor map: a kernel argument of the d = 128 square pass only (the
// others store O with plain stores, and a larger argument block measured
// slower on short launches).
template <bool kHave>
struct OMapArg {
  CUtensorMap map;
};
template <>
struct OMapArg<false> {};

// Work tile u (0 <= u < BH * num_mblocks) is m-block r = u / BH of head
// bh = u % BH, m-blocks heaviest first under the causal mask.  CTA c of G
// takes tiles in rounds of G: round k gives it tile k*G + c, or k*G + G-1-c
// on odd rounds, so the heavy and light ends of each round even out.
__device__ __forceinline__ int fwd_tile_of_round(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Zeroes the split pass's work-tile counter before each call.  The split
// pass is launched as its programmatic dependent, so that pass's CTAs set up
// while this one-thread kernel runs.
__global__ void split_counter_reset_kernel(int* counter) {
  ptx::griddep_launch_dependents();
  *counter = 0;
}

// SPLIT = false: the attention forward pass (square, top-left causal mask).
// SPLIT = true: the partial pass of split-KV decoding (bottom-right causal
// mask, fp32 partial outputs for splitkv_merge_kernel); a split's K/V tiles
// alternate between the two stages, each of which writes a partial of its
// own, the Q buffers of both stages serve as two Q sets, and work tiles are
// handed out at run time.
// PAGED = true (with SPLIT): the same pass over a paged K/V cache, each
// batch entry with its own key count; tmK / tmV then map the cache
// [blocks][heads][page rows][d] with boxes of min(page_size, 128) rows: at
// d = 64 as 4-D [blocks][heads][page rows][d]; at d = 128 as 5-D
// [blocks * heads][8-row group][d-half][row][64], which brings both
// d-halves of a box's rows in one copy.
template <int D, bool CAUSAL, bool SPLIT = false, bool PAGED = false, bool HMAJOR = false>
__global__ void __launch_bounds__(FwdCfg<D, SPLIT>::kThreads, 1)
    mha_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ OMapArg<FwdCfg<D, SPLIT>::kOSets != 0> tmO, const FwdParams p) {
  using C = FwdCfg<D, SPLIT>;
  static_assert(SPLIT || !PAGED, "the paged pass is a split pass");
  static_assert(!(SPLIT && HMAJOR), "the head-major order is one of the square pass");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = SPLIT ? p.Nk : p.N;  // keys (and, square, queries)
  const int n_tiles = (N + C::kBlockN - 1) / C::kBlockN;
  const int total = p.BH * (SPLIT ? p.num_splits : p.num_mblocks);
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  // K/V tiles each Q tile needs (0 when the Q tile lies past the end).
  auto tiles_for = [&](int row0) {
    return row0 >= N ? 0 : (CAUSAL ? min(n_tiles, row0 / C::kBlockN + 1) : n_tiles);
  };
  // a work tile: head, first query row, K/V tiles per stage and in all,
  // keys of the head (split mode: nkv is 0 for a split past them)
  struct Tile {
    int bh, m0, n0, n1, nkv, kv_begin, split, nk;
  };
  // split mode: tile u is split u / BH of head bh = u % BH, so the heads of
  // one batch entry (bh = b * heads + h) are adjacent.  Every tile runs on
  // stage 0 (running odd tiles on stage 1, so that one tile's epilogue
  // overlaps the next one's start, measured 2-3% slower).
  auto keys_of = [&](int bh) {
    return PAGED ? max(0, min(p.seq_lens[bh / p.num_heads], p.max_blocks * p.page_size)) : N;
  };
  auto split_tile = [&](int u, Tile& t) {
    t.bh = u % p.BH;
    t.split = u / p.BH;
    t.kv_begin = t.split * p.tiles_per_split;
    t.m0 = 0;
    t.nk = keys_of(t.bh);
    // the split's K/V tiles alternate between the stages: stage s takes
    // tiles j = s mod 2
    t.nkv = max(0, min(p.tiles_per_split, (t.nk + C::kBlockN - 1) / C::kBlockN - t.kv_begin));
    t.n0 = (t.nkv + 1) / 2;
    t.n1 = t.nkv / 2;
  };
  // square mode: the k-th tile of this CTA in the static order
  auto tile_at = [&](int k, Tile& t) -> bool {
    t.nk = N;
    t.split = 0;
    t.kv_begin = 0;
    if constexpr (HMAJOR) {
      // Head-major order: CTA c takes items c, c + G, c + 2G, ...; the items
      // of one head are adjacent, so the grid works on a few heads' K/V at a
      // time and they stay in L2.  Under the causal mask item i of a head is
      // the pair of m-blocks M-1-i (first) and i, whose K/V tile counts add
      // up to the same M + 1 for every pair, so the rounds stay balanced; the
      // middle m-block of an odd M has no partner, and its second tile is
      // empty (placed past the end).
      const int per_head = CAUSAL ? (p.num_mblocks + 1) >> 1 : p.num_mblocks;
      const int w = c + (CAUSAL ? (k >> 1) : k) * G;
      if (w >= p.BH * per_head) return false;
      t.bh = w / per_head;
      const int i = w - t.bh * per_head;
      int mblk = i;
      bool empty = false;
      if constexpr (CAUSAL) {
        const int hi = p.num_mblocks - 1 - i;
        mblk = (k & 1) ? i : hi;
        empty = (k & 1) && hi == i;
      }
      t.m0 = empty ? N : mblk * 256;
    } else {
      const int u = fwd_tile_of_round(k, c, G);
      if (u >= total) return false;
      t.bh = u % p.BH;
      const int r = u / p.BH;
      const int mblk = CAUSAL ? (p.num_mblocks - 1 - r) : r;
      t.m0 = mblk * 256;
    }
    t.n0 = tiles_for(t.m0);
    t.n1 = tiles_for(t.m0 + C::kBlockM);
    t.nkv = max(t.n0, t.n1);  // both stages read the same K/V tiles
    return true;
  };

  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  // Q set b holds work tiles b, b + kQS, ...: the m-th use of a set is
  // phase m of its barriers.  Split mode needs one Q tile per work tile,
  // so the buffers of both stages make two sets.
  constexpr int kQS = SPLIT ? 2 : C::kQSets;
  auto q_full = [&](int b) { return bar(b); };       // the work tile's Q tiles loaded
  auto q_empty = [&](int b) { return bar(2 + b); };  // every S MMA reading them done
  auto q_set = [](int k) { return k % kQS; };
  auto q_par = [](int k) { return (k / kQS) & 1; };
  auto kv_full = [&](int i) { return bar(4 + i); };
  auto kv_empty = [&](int i) { return bar(4 + C::kStages + i); };
  auto s_full = [&](int s) { return bar(4 + 2 * C::kStages + s); };
  auto p_ready = [&](int s) { return bar(6 + 2 * C::kStages + s); };
  auto o_full = [&](int s) { return bar(8 + 2 * C::kStages + s); };
  const uint32_t drain_bar = bar(10 + 2 * C::kStages);
  const uint32_t tail_bar = bar(11 + 2 * C::kStages);
  auto tile_full = [&](int i) { return bar(12 + 2 * C::kStages + i); };
  auto tile_empty = [&](int i) { return bar(12 + 2 * C::kStages + C::kTileRing + i); };
  auto o_free = [&](int i) { return bar(12 + 2 * C::kStages + 2 * C::kTileRing + i); };
  int* tile_ids = reinterpret_cast<int*>(smem + C::kOffTileIds);
  // Q tile of set b, stage s
  auto q_index = [](int b, int s) { return SPLIT ? b : 2 * b + s; };
  auto sQ = [&](int b, int s) -> uint32_t { return sbase + C::kOffQ + q_index(b, s) * C::kTileBytes; };
  auto sKV = [&](int i) -> uint32_t { return sbase + C::kOffKV + i * C::kTileBytes; };
  // Layout of a K/V tile in shared memory: 8-key groups of 128-byte swizzle
  // atoms.  Contiguous K/V: each d-half is a 16 KiB block of its own (groups
  // 1 KiB apart).  Paged at d = 128: one copy per page brings both halves
  // of its keys, so a group holds its two atoms side by side (halves 1 KiB
  // apart, groups 2 KiB apart); the tensor core reads either through the
  // same descriptors with these two strides.
  constexpr bool kPairedHalves = PAGED && D == 128;
  constexpr int kKVGroupBytes = kPairedHalves ? 2048 : 1024;
  constexpr int kKVHalfBytes = kPairedHalves ? 1024 : C::kHalfBytes;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit};

  // The k-th work tile of this CTA, for every role but the K/V producer.
  // Square mode: the static order.  Split mode: the k-th id the K/V
  // producer put in the ring (an id >= total ends the work).  One thread
  // (warp_wide false) or a whole warp calls it; false at the end of the
  // work, or with ok = false when a wait gave up.
  auto take_tile = [&](int k, Tile& t, bool& ok, bool warp_wide, unsigned site) -> bool {
    if constexpr (!SPLIT) {
      return tile_at(k, t);
    } else {
      const int slot = k % C::kTileRing;
      const uint32_t par = (k / C::kTileRing) & 1;
      if (!(warp_wide ? wait_warp(tile_full(slot), par, ctl, site) : wait_one(tile_full(slot), par, ctl, site))) {
        ok = false;
        return false;
      }
      const int u = tile_ids[slot];
      if (warp_wide) __syncwarp();
      if (!warp_wide || lane == 0) ptx::mbar_arrive(tile_empty(slot));
      if (u >= total) return false;
      split_tile(u, t);
      return true;
    }
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(q_full(b), 1);
      ptx::mbar_init(q_empty(b), 1);
    }
    for (int i = 0; i < C::kStages; ++i) {
      ptx::mbar_init(kv_full(i), 1);
      ptx::mbar_init(kv_empty(i), 1);
    }
    // one elected arrive per softmax warp of the stage; split mode: the
    // Nq <= 32 query rows lie in the first warp of each stage, and the other
    // softmax warps have no work there and wait at the final barrier
    const int p_arrivals = SPLIT ? 1 : 4;
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(s_full(s), 1);
      ptx::mbar_init(p_ready(s), p_arrivals);
      ptx::mbar_init(o_full(s), 1);
    }
    ptx::mbar_init(drain_bar, 1);
    ptx::mbar_init(tail_bar, 1);
    for (int i = 0; i < C::kTileRing; ++i) {
      ptx::mbar_init(tile_full(i), 1);
      ptx::mbar_init(tile_empty(i), 2 + 2 * p_arrivals);  // one arrive per consumer warp
    }
    for (int i = 0; i < 4; ++i) ptx::mbar_init(o_free(i), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmQ);
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
    if constexpr (C::kOSets > 0) ptx::prefetch_tensormap(&tmO.map);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if constexpr (C::kSumCol) {
    // the ones tile in the V tiles' layout (MN-major, 128-byte swizzle): key
    // k's row holds bf16 1.0 at N-position 0 of the atom, i.e. in 16-byte
    // piece 0 ^ (k mod 8), and zeros elsewhere; thread k < 128 writes row k
    if (threadIdx.x < 128) {
      const int k = threadIdx.x;
      uint4* row = reinterpret_cast<uint4*>(smem + C::kOffOnes + (k >> 3) * 1024 + (k & 7) * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) row[c] = make_uint4(c == (k & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
      ptx::fence_proxy_async_smem();  // read by the tensor core
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // split mode: the merge kernel may start on SMs this grid leaves (it
  // waits for this grid's completion before reading any partial).  This
  // grid is itself a dependent of split_counter_reset_kernel: the set-up
  // above overlaps that kernel, and nothing below runs before it and all
  // work queued ahead of it have completed.
  if constexpr (SPLIT) {
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    ptx::griddep_wait();
  }

  if (warp == 0) {
    // -------------------------------------------------- K/V producer
    // K_j, V_j of every work tile in turn through one ring; position t
    // runs on across work tiles.  The whole warp walks the loop (its waits
    // stay warp-uniform) and one lane issues the copies.
    int t = 0;
    int scrubs = 0;  // tail_bar phases used
    bool ok = true;
    // paged mode: a K or V tile is `chunks` boxes of `rows` keys, each from
    // the page its first key lies in; lane r < chunks issues box r.  Each
    // lane reads its block id one K/V tile ahead (and the first one of the
    // next work tile while this one's last copies land), so the table's
    // latency overlaps the ring waits instead of adding to them.
    const int rows = PAGED ? min(p.page_size, C::kBlockN) : C::kBlockN;
    const int chunks = C::kBlockN / rows;
    auto block_of = [&](const Tile& w, int j) -> int {
      const int pos = (w.kv_begin + j) * C::kBlockN + lane * rows;
      // a page past the entry's length reads as zeros (a block id past the
      // cache); pos < nk also keeps the table read inside its row
      if (lane >= chunks || pos >= w.nk) return p.num_blocks;
      const int b = p.block_table[static_cast<size_t>(w.bh / p.num_heads) * p.max_blocks + pos / p.page_size];
      // any other id outside the cache reads as zeros too; clamping it keeps
      // block * heads + head inside int for the 5-D map
      return static_cast<unsigned>(b) < static_cast<unsigned>(p.num_blocks) ? b : p.num_blocks;
    };
    // split mode: this warp draws the work tiles (the first one is the
    // CTA's index, each further one comes from the global counter once the
    // current tile's last copy is issued) and hands their ids to the other
    // roles through the ring
    int published = 0;
    auto publish = [&](int u) -> bool {
      const int slot = published % C::kTileRing;
      if (published >= C::kTileRing &&
          !wait_warp(tile_empty(slot), ((published / C::kTileRing) - 1) & 1, ctl, kSiteProducerEmpty))
        return false;
      if (lane == 0) {
        tile_ids[slot] = u;
        ptx::mbar_arrive(tile_full(slot));  // release: the id is visible to whoever sees the phase
      }
      __syncwarp();
      ++published;
      return true;
    };
    auto empty_split = [&](int u) {
      return (u / p.BH) * p.tiles_per_split * C::kBlockN >= keys_of(u % p.BH);
    };
    auto draw = [&]() -> int {
      int u = 0;
      if (lane == 0) {
        u = G + atomicAdd(p.tile_counter, 1);
        if constexpr (PAGED) {
          // a split past an entry's keys is past them for every head of the
          // entry: move the counter beyond that run of heads
          while (u < total && empty_split(u)) {
            atomicMax(p.tile_counter, u - u % p.num_heads + p.num_heads - G);
            u = G + atomicAdd(p.tile_counter, 1);
          }
        }
      }
      return __shfl_sync(0xffffffffu, u, 0);
    };
    Tile tl;
    bool have;
    if constexpr (SPLIT) {
      int u = c;
      if (PAGED && empty_split(u)) u = draw();
      ok = publish(u);
      have = ok && u < total;
      if (have) split_tile(u, tl);
    } else {
      have = tile_at(0, tl);
    }
    int blk_next = (PAGED && have) ? block_of(tl, 0) : 0;
    for (int k = 0; ok && have; ++k) {
      const int n_kv = tl.nkv;
      // split mode: the next tile is drawn once this one's last copy is
      // issued (drawing it two K/V tiles earlier measured the same)
      int u_next = total;
      if (SPLIT && n_kv == 0) {
        u_next = draw();
        ok = publish(u_next);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int key0 = (tl.kv_begin + j) * C::kBlockN;
        const int blk = blk_next;
        if (PAGED && j + 1 < n_kv) blk_next = block_of(tl, j + 1);
        for (int which = 0; which < 2; ++which, ++t) {
          const int slot = t % C::kStages;
          const int use = t / C::kStages;
          if (use > 0 && !wait_warp(kv_empty(slot), (use - 1) & 1, ctl, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const CUtensorMap* map = which ? &tmV : &tmK;
          if constexpr (PAGED) {
            // every box lands 1 KiB aligned, so the 128-byte swizzle of the
            // tile is that of one 128-row box
            const int valid = tl.nk - key0;  // keys of this tile inside the entry (>= 1)
            // V rows past the entry's length that come from its last,
            // partly filled page hold whatever the cache holds there,
            // possibly NaN, and a zero weight times NaN is NaN: that copy
            // lands on tail_bar, the rows get cleared, and only then is the
            // slot marked full (masked scores make the same rows of K harmless)
            const bool scrub = which == 1 && valid < C::kBlockN && valid % rows != 0;
            const uint32_t done = scrub ? tail_bar : kv_full(slot);
            if (lane == 0) ptx::mbar_arrive_expect_tx(done, C::kTileBytes);
            __syncwarp();
            if (lane < chunks) {
              const int head = tl.bh % p.num_heads;
              const int pos = key0 + lane * rows;
              if constexpr (kPairedHalves) {
                // 5-D map [block * heads + head][8-key group][half][key][64]
                ptx::tma_load_5d(sKV(slot) + lane * rows * 256, map, done, 0, 0, 0,
                                 (pos % p.page_size) / 8, blk * p.num_heads + head);
              } else {
                for (int h = 0; h < C::kHalves; ++h)
                  ptx::tma_load_4d(sKV(slot) + h * C::kHalfBytes + lane * rows * 128, map, done, h * 64,
                                   pos % p.page_size, head, blk);
              }
            }
            __syncwarp();
            if (scrub) {
              if (!wait_warp(tail_bar, scrubs & 1, ctl, kSiteProducerEmpty)) {
                if (lane == 0) drain_wait(tail_bar, scrubs & 1, ctl);
                ok = false;
                break;
              }
              ++scrubs;
              uint8_t* vt = smem + C::kOffKV + slot * C::kTileBytes;
              // 16-byte pieces of keys valid..127: 8 per key and half
              constexpr int kPerKey = 8 * C::kHalves;
              for (int i = lane; i < (C::kBlockN - valid) * kPerKey; i += 32) {
                const int key = valid + i / kPerKey, r = i % kPerKey;
                *reinterpret_cast<uint4*>(vt + (key / 8) * kKVGroupBytes + (r / 8) * kKVHalfBytes +
                                          (key % 8) * 128 + (r % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
              }
              ptx::fence_proxy_async_smem();  // visible to the tensor core's reads
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(kv_full(slot));
            }
          } else {
            if (lane == 0) {
              ptx::mbar_arrive_expect_tx(kv_full(slot), C::kTileBytes);
              for (int h = 0; h < C::kHalves; ++h)
                ptx::tma_load_3d(sKV(slot) + h * C::kHalfBytes, map, kv_full(slot), h * 64, key0, tl.bh);
            }
            __syncwarp();
          }
        }
        if (SPLIT && ok && j == n_kv - 1) {
          u_next = draw();
          ok = publish(u_next);
        }
      }
      if (!ok) break;
      if constexpr (SPLIT) {
        have = u_next < total;
        if (have) split_tile(u_next, tl);
      } else {
        have = tile_at(k + 1, tl);
      }
      if (PAGED && have) blk_next = block_of(tl, 0);
    }
    if (!ok && lane == 0) {
      // let the copies already issued land before the CTA goes away
      for (int u = max(0, t - C::kStages); u < t; ++u)
        drain_wait(kv_full(u % C::kStages), (u / C::kStages) & 1, ctl);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------ Q producer
    // The next work tile's Q goes in as soon as the tensor core has run the
    // current tile's last Q K^T, overlapping that tile's last softmax and
    // epilogue.
    if (lane == 0) {
      Tile tl;
      int kq = 0;  // work tiles with K/V tiles so far: the sets go to those only
      bool ok = true;
      for (int k = 0; ok && take_tile(k, tl, ok, false, kSiteProducerEmpty); ++k) {
        if (tl.nkv == 0) continue;  // a split past the head's keys
        // the set's previous tile (kq - kQSets) must be done with it
        const int prev = kq - kQS;
        if (prev >= 0 && !wait_one(q_empty(q_set(prev)), q_par(prev), ctl, kSiteProducerEmpty)) {
          ok = false;
          break;
        }
        const int b = q_set(kq);
        const int stages = (!SPLIT && tl.n1 > 0) ? 2 : 1;  // split mode: one Q tile
        ptx::mbar_arrive_expect_tx(q_full(b), stages * C::kTileBytes);
        for (int s = 0; s < stages; ++s)
          for (int h = 0; h < C::kHalves; ++h)
            ptx::tma_load_3d(sQ(b, s) + h * C::kHalfBytes, &tmQ, q_full(b), h * 64,
                             tl.m0 + s * C::kBlockM, tl.bh);
        ++kq;
      }
      if (!ok)
        for (int u = max(0, kq - kQS); u < kq; ++u) drain_wait(q_full(q_set(u)), q_par(u), ctl);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, C::kBlockN, 0, 0);
      constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(128, C::kONcols, 0, 1);
      const uint32_t tS0 = tmem + C::kColS0, tS1 = tmem + C::kColS1;
      const uint32_t tO0 = tmem + C::kColO0, tO1 = tmem + C::kColO1;
      // Descriptors are built once; moving to another slot or k-step only
      // adds (byte offset >> 4) to the start-address field, which never
      // carries out of it because every operand lies below 256 KiB.  The
      // single issuing thread is the tensor core's only feeder, so keeping
      // its per-MMA work to an add and the instruction itself matters.
      // Every lane of the warp runs this loop with the same values; that
      // keeps them warp-uniform, and an elected lane issues.
      // Q and K tiles: K-major, 128-byte swizzle, 8-row groups (SBO) 1 KiB
      // apart (K: kKVGroupBytes).
      const uint64_t dQ00 = ptx::desc_sw128(sQ(0, 0), 16, 1024);
      const uint64_t dK0 = ptx::desc_sw128(sKV(0), 16, kKVGroupBytes);
      // V tiles: MN-major (d contiguous), d-halves kKVHalfBytes apart (LBO),
      // 8-key groups kKVGroupBytes apart (SBO).
      // With the sum column, N-atom 1 of every slot's V is the ones tile: the
      // stride field holds (ones - slot) >> 4, so moving to slot i adds
      // i * tile >> 4 to the start field and takes it off the stride field
      // (which stays positive: the ones tile lies past the ring).
      const uint64_t dV0 =
          ptx::desc_sw128(sKV(0), C::kSumCol ? sbase + C::kOffOnes - sKV(0) : kKVHalfBytes, kKVGroupBytes);
      auto slot_off = [](int slot) -> uint64_t {
        return static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
      };
      auto v_off = [](int slot) -> uint64_t {
        const uint64_t a = static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
        return C::kSumCol ? a - (a << 16) : a;
      };
      // S(s) = Q_s K^T over K = d in steps of 16
      auto issue_s = [&](int qb, int s, int kslot) {
        const uint64_t dk = dK0 + slot_off(kslot);
        const uint64_t dq = dQ00 + static_cast<uint64_t>((q_index(qb, s) * C::kTileBytes) >> 4);
        const uint32_t ts = s ? tS1 : tS0;
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t qoff =
                static_cast<uint64_t>(((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4);
            const uint64_t koff =
                static_cast<uint64_t>(((kk >> 2) * kKVHalfBytes + (kk & 3) * 32) >> 4);
            ptx::mma_ss(ts, dq + qoff, dk + koff, kIdescS, kk > 0 ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      // O(so) += P V over 128 keys in steps of 16; P read from TMEM, from
      // the S columns of stage sp
      auto issue_pv_from = [&](int sp, int so, int vslot, bool first) {
        const uint64_t dv = dV0 + v_off(vslot);
        const uint32_t ts = sp ? tS1 : tS0;
        const uint32_t to = so ? tO1 : tO0;
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < C::kBlockN / 16; ++kk)
            ptx::mma_ts(to, ts + kk * 8, dv + static_cast<uint64_t>((kk * 2 * kKVGroupBytes) >> 4),
                        kIdescO, (!first || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int s, int vslot, bool first) { issue_pv_from(s, s, vslot, first); };
      auto commit = [&](uint32_t b) {
        if (ptx::elect_one()) ptx::mma_commit(b);
        __syncwarp();
      };
      bool ok = true;
      int t = 0;                 // K/V ring position
      int pr[2] = {0, 0};        // p_ready completions consumed, per stage
      Tile tl;
      int kq = 0;                // work tiles with K/V tiles so far (Q set uses)
      for (int k = 0; ok && take_tile(k, tl, ok, true, kSiteMmaQ); ++k) {
        auto n_s = [&](int s) { return s ? tl.n1 : tl.n0; };
        const int n_kv = tl.nkv;
        if (n_kv == 0) continue;  // a split past the head's keys
        const int qb = q_set(kq);
        if (!(ok = wait_warp(q_full(qb), q_par(kq), ctl, kSiteMmaQ))) break;
        ++kq;
        if constexpr (SPLIT) {
          // The split's K/V tiles alternate between the stages (stage s
          // takes tiles j = s mod 2, with its own S columns, O accumulator
          // and softmax warp), and S_{j+1} is issued before P_j V_j: the two
          // softmax warps work on consecutive tiles at the same time, and
          // neither waits for P V before its next scores.  The MMAs run in
          // issue order, so S_{j+2} overwrites P_j only after P_j V_j, and
          // when a stage sees S_j complete its P_{j-2} V_{j-2} is done too.
          const int n = tl.nkv;
          const int t0 = t;  // ring position of K_0
          auto slot_of = [&](int pos) { return pos % C::kStages; };
          auto par_of = [&](int pos) { return static_cast<uint32_t>((pos / C::kStages) & 1); };
          for (int j = -1; j < n && ok; ++j) {
            if (j + 1 < n) {
              const int kp = t0 + 2 * (j + 1);  // K_{j+1}
              if (!(ok = wait_warp(kv_full(slot_of(kp)), par_of(kp), ctl, kSiteMmaKV))) break;
              ptx::tc_fence_after();
              issue_s(qb, (j + 1) & 1, slot_of(kp));
              commit(s_full((j + 1) & 1));
              commit(kv_empty(slot_of(kp)));
              if (j + 2 == n) commit(q_empty(qb));  // this tile's Q is no longer read
            }
            if (j < 0) continue;
            const int st = j & 1;
            const int vp = t0 + 2 * j + 1;  // V_j
            // (pr indexed with constants only, so that it stays in registers)
            const int seen = st ? pr[1] : pr[0];
            if (!(ok = wait_warp(p_ready(st), seen & 1, ctl, kSiteMmaP))) break;
            if (st) ++pr[1]; else ++pr[0];
            if (!(ok = wait_warp(kv_full(slot_of(vp)), par_of(vp), ctl, kSiteMmaKV))) break;
            ptx::tc_fence_after();
            issue_pv(st, slot_of(vp), j < 2);
            if (j >= n - 2) commit(o_full(st));  // the stage's last tile of this split
            commit(kv_empty(slot_of(vp)));
          }
          t = t0 + 2 * n;
          continue;
        }
        int v_prev = 0;
        for (int j = 0; j < n_kv && ok; ++j) {
          const int k_slot = t % C::kStages, k_par = (t / C::kStages) & 1;
          ++t;
          const int v_slot = t % C::kStages, v_par = (t / C::kStages) & 1;
          ++t;
          if (!(ok = wait_warp(kv_full(k_slot), k_par, ctl, kSiteMmaKV))) break;
          ptx::tc_fence_after();
          for (int s = 0; s < 2 && ok; ++s) {
            if (j >= 1 && j - 1 < n_s(s)) {
              if (!(ok = wait_warp(p_ready(s), pr[s] & 1, ctl, kSiteMmaP))) break;
              ++pr[s];
              ptx::tc_fence_after();
              issue_pv(s, v_prev, j - 1 == 0);
              if (j - 1 == n_s(s) - 1) commit(o_full(s));
            }
            if (j < n_s(s)) {
              issue_s(qb, s, k_slot);
              commit(s_full(s));
            }
          }
          if (!ok) break;
          if (j == n_kv - 1) commit(q_empty(qb));  // this tile's Q is no longer read
          commit(kv_empty(k_slot));
          if (j >= 1) commit(kv_empty(v_prev));
          if (!(ok = wait_warp(kv_full(v_slot), v_par, ctl, kSiteMmaKV))) break;
          ptx::tc_fence_after();
          v_prev = v_slot;
        }
        for (int s = 0; s < 2 && ok; ++s) {
          if (n_kv - 1 < n_s(s)) {
            if (!(ok = wait_warp(p_ready(s), pr[s] & 1, ctl, kSiteMmaP))) break;
            ++pr[s];
            ptx::tc_fence_after();
            issue_pv(s, v_prev, n_kv - 1 == 0);
            commit(o_full(s));
          }
        }
        if (ok) commit(kv_empty(v_prev));
      }
      // every MMA this warp issued completes before TMEM is released
      commit(drain_bar);
      if (lane == 0) drain_wait(drain_bar, 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------- softmax / correction
    const int s = (warp - 4) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + (s ? C::kColS1 : C::kColS0);
    const uint32_t t_o = tmem + lane_off + (s ? C::kColO1 : C::kColO0);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int sf = 0;  // s_full completions consumed
    int of = 0;  // o_full completions consumed
    int ouse = 0;  // square mode: epilogues on this warp's staging chunk so far
    Tile tl;
    // split mode: the Nq <= 32 query rows lie in the first warp of each
    // stage; the other softmax warps have no work and go straight to the
    // final barrier (not even polling the tile ring), which leaves their SM
    // sub-partitions to the warps that share them
    const bool idle = SPLIT && wq > 0;
    for (int k = 0; !idle && ok && take_tile(k, tl, ok, true, kSiteSoftmaxS); ++k) {
      const int m0 = tl.m0;
      const int n = s ? tl.n1 : tl.n0;
      const int q_idx = SPLIT ? row : m0 + s * C::kBlockM + row;
      // square mode: this work tile's use of the staging chunk (d = 128:
      // the chunk is shared, stage 0's epilogue of a work tile comes first)
      int my_use = 0;
      if constexpr (C::kOSets > 0) {
        my_use = ouse + ((s == 1 && tl.n0 > 0) ? 1 : 0);
        ouse += (tl.n0 > 0 ? 1 : 0) + (tl.n1 > 0 ? 1 : 0);
      }
      float m_run = -INFINITY;  // running max of scale*log2(e)*s, possibly stale
      float l_run = 0.f;   // row sum of exp2 terms (fp32), for the LSE
      float lr_run = 0.f;  // the same over the bf16-rounded terms, for O
      for (int j = 0; j < n; ++j) {
        if (!wait_warp(s_full(s), sf & 1, ctl, kSiteSoftmaxS)) {
          ok = false;
          break;
        }
        ++sf;
        ptx::tc_fence_after();
        uint32_t raw[128];
        ptx::tmem_ld_x128(t_s, raw);
        float x[128];
#pragma unroll
        for (int cc = 0; cc < 128; ++cc) x[cc] = __uint_as_float(raw[cc]);
        // this stage's j-th K/V tile (split mode: tile 2j + s of the split)
        const int kv0 = (tl.kv_begin + (SPLIT ? 2 * j + s : j)) * C::kBlockN;
        const int nk = tl.nk;  // keys of this head
        // square: query i sees keys 0..i; split: query i of Nq sees keys
        // 0..nk-Nq+i (the queries are the last Nq positions)
        const int diag = SPLIT ? nk - p.Nq : m0 + s * C::kBlockM;  // first row's last visible key
        const bool edge = (kv0 + C::kBlockN > nk) || (CAUSAL && kv0 + C::kBlockN - 1 > diag);
        if (edge) {
          const int last = SPLIT ? nk - p.Nq + q_idx : q_idx;  // this row's last visible key
          const int lim = (CAUSAL ? min(nk, last + 1) : nk) - kv0;  // keys [kv0, kv0+lim) visible
#pragma unroll
          for (int cc = 0; cc < 128; ++cc)
            if (cc >= lim) x[cc] = -INFINITY;
        }
        // row maximum of this tile: 8 independent chains of 3-input max
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
        for (int cc = 8; cc < 128; cc += 2) mx[(cc >> 1) & 7] = ptx::max3(mx[(cc >> 1) & 7], x[cc], x[cc + 1]);
        const float tile_max = fmaxf(ptx::max3(mx[0], mx[1], mx[2]),
                                     fmaxf(ptx::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_tile = tile_max * sl2;
        float alpha = 1.f;
        if (m_tile > m_run + C::kRescaleThreshold) {
          alpha = (m_run == -INFINITY) ? 0.f : ptx::ex2(m_run - m_tile);
          m_run = m_tile;
        }
        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negm = make_float2(neg_m, neg_m);
        float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // fp32 p: for the LSE
        float sumr[4] = {0.f, 0.f, 0.f, 0.f};  // bf16 p: for O / l
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 tt = __ffma2_rn(make_float2(x[c4 * 32 + 2 * i], x[c4 * 32 + 2 * i + 1]), sl2v, negm);
            const float p0 = ptx::ex2(tt.x);
            const float p1 = ptx::ex2(tt.y);
            pk[i] = ptx::pack_bf16x2(p0, p1);
            sum2[i & 1] = __fadd2_rn(sum2[i & 1], make_float2(p0, p1));
            // normalising O by the sum of the bf16 values the tensor core
            // multiplies into V keeps O an exact convex combination of V rows
            // (a row that one key dominates reproduces that key's V row even
            // when the running max is stale and that key's P is rounded)
            if constexpr (!C::kSumCol) {
              sumr[(2 * i) & 3] = ptx::add_bf16_lo(pk[i], sumr[(2 * i) & 3]);
              sumr[(2 * i + 1) & 3] = ptx::add_bf16_hi(pk[i], sumr[(2 * i + 1) & 3]);
            }
          }
          ptx::tmem_st_x16(t_s + c4 * 16, pk);
        }
        l_run = l_run * alpha + ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y));
        lr_run = lr_run * alpha + ((sumr[0] + sumr[1]) + (sumr[2] + sumr[3]));
        // correction: bring O(s) to the new max before P_j(s) V_j lands on it
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            ptx::tmem_ld_x32(t_o + cc * 32, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            ptx::tmem_st_x32(t_o + cc * 32, ov);
          }
          if constexpr (C::kSumCol)
            ptx::tmem_st_x1(t_o + D, __float_as_uint(__uint_as_float(ptx::tmem_ld_x1(t_o + D)) * alpha));
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_ready(s));
      }
      if (!ok) continue;
      if constexpr (SPLIT) {
        if (n == 0) {
          // a one-tile split leaves stage 1 without keys: an empty partial
          // (the merge gives it zero weight; its O must still be finite)
          if (q_idx < p.Nq) {
            const size_t prow =
                (static_cast<size_t>(tl.bh) * 2 * p.num_splits + 2 * tl.split + s) * p.Nq + q_idx;
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
            for (int v4 = 0; v4 < D / 4; ++v4) dst[v4] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse_part[prow] = -INFINITY;
          }
          continue;
        }
      }
      if (n == 0) continue;
      if (!wait_warp(o_full(s), of & 1, ctl, kSiteSoftmaxO)) {
        ok = false;
        break;
      }
      ++of;
      ptx::tc_fence_after();
      // epilogue: O = O_acc / l in bf16, LSE = (m + log2 l) * ln 2.  The next
      // work tile's first P V overwrites O(s) only after this warp's next
      // p_ready arrival, which follows these reads.
      if constexpr (C::kSumCol) lr_run = __uint_as_float(ptx::tmem_ld_x1(t_o + D));  // the tensor core's sum
      const float inv_l = lr_run > 0.f ? 1.f / lr_run : 0.f;
      const float m_fin = (m_run == -INFINITY) ? 0.f : m_run;
      const float lse_row = l_run > 0.f ? (m_fin + log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
      if constexpr (SPLIT) {
        // fp32 partial row of this stage's half of the split, normalised by
        // its own sum: each split gives two partials, 2 * split + stage.  The
        // TMEM loads are warp-collective: every lane issues them, only rows
        // below Nq store.
        const bool live = q_idx < p.Nq;
        const size_t prow =
            (static_cast<size_t>(tl.bh) * 2 * p.num_splits + 2 * tl.split + s) * p.Nq + (live ? q_idx : 0);
        float* orow = p.o_part + prow * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          ptx::tmem_ld_x32(t_o + cc * 32, ov);
          if (live) {
            float4* dst = reinterpret_cast<float4*>(orow + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(ov[4 * v4]) * inv_l, __uint_as_float(ov[4 * v4 + 1]) * inv_l,
                                    __uint_as_float(ov[4 * v4 + 2]) * inv_l, __uint_as_float(ov[4 * v4 + 3]) * inv_l);
          }
        }
        if (live) p.lse_part[prow] = lse_row;
        ptx::tc_fence_before();
        continue;
      }
      if constexpr (C::kOSets > 0) {
        // square mode: O / l in bf16 into this warp's staging chunk, laid out
        // as the O tensor map's 128-byte swizzle expects (16-byte piece c of
        // row r at position c ^ (r mod 8) of the row), then one TMA store per
        // d-half of the warp's 32 rows; rows past N are not written
        const uint32_t chunk = sbase + C::kOffO + wq * C::kOChunkBytes;
        // the other stage's warp on this lane quarter is done with the chunk
        if (my_use > 0 && !wait_warp(o_free(wq), (my_use - 1) & 1, ctl, kSiteSoftmaxO)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          ptx::tmem_ld_x32(t_o + cc * 32, ov);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = ptx::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                     __uint_as_float(ov[2 * i + 1]) * inv_l);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int piece = cc * 4 + v4;  // 16-byte piece (8 columns) of the row
            const uint32_t addr = chunk + (piece >> 3) * 4096 + lane * 128 + (((piece & 7) ^ (lane & 7)) << 4);
            ptx::st_shared_v4(addr, pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        ptx::fence_proxy_async_smem();  // the chunk is read by the async proxy
        __syncwarp();
        const int row0 = m0 + s * C::kBlockM + wq * 32;  // this warp's first row
        if (lane == 0) {
          if (row0 < N) {
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) ptx::tma_store_3d(&tmO.map, chunk + h * 4096, h * 64, row0, tl.bh);
            ptx::bulk_commit_group();
          }
          ptx::bulk_wait_read_all();
          ptx::mbar_arrive(o_free(wq));
        }
        __syncwarp();
      } else {
        const bool valid = q_idx < N;
        __nv_bfloat16* orow = p.o + (static_cast<size_t>(tl.bh) * N + (valid ? q_idx : 0)) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          ptx::tmem_ld_x32(t_o + cc * 32, ov);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = ptx::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                     __uint_as_float(ov[2 * i + 1]) * inv_l);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
      }
      if (q_idx < N) p.lse[static_cast<size_t>(tl.bh) * N + q_idx] = lse_row;
      ptx::tc_fence_before();
    }
    // the O stores complete before the CTA (and its shared memory) goes away
    if (C::kOSets > 0 && lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// One warp waits, with the kernel's bounded wait, on a barrier nothing ever
// completes; the wait must give up, record a timeout and return.
__global__ void wait_selftest_kernel(unsigned* status, long long limit) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, status, limit};
  wait_warp(b, 0, ctl, kSiteSelftest);
  __syncwarp();
}

}  // namespace mha
