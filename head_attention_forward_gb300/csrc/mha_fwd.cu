// mha_fwd.cu - host side of the attention library: argument checks, TMA
// tensor maps, launch configuration and the extern "C" entry points that
// include/mha_fwd.h declares.
//
// The library links the CUDA runtime statically and reaches the one driver
// entry point it needs (cuTensorMapEncodeTiled) through the runtime, so the
// shared object loads on machines without a GPU driver; every entry point
// validates its arguments before touching CUDA.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "mha_fwd.h"
#include "mha_fwd_kernel.cuh"
#include "mha_internal.h"

namespace {

// One status word per device (module memory, not an allocation).
__device__ unsigned g_status;

constexpr int kMaxDevices = 64;
constexpr long long kDefaultWaitLimit = 1ll << 31;

std::mutex g_mu;
long long g_wait_limit = kDefaultWaitLimit;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct DeviceState {
  bool ready = false;
  bool ok = false;
  unsigned* status = nullptr;
  int sms = 0;  // multiprocessor count: the persistent grid's size
};
DeviceState g_dev[kMaxDevices];

}  // namespace

namespace mha_host {

// Per-device set-up, done once under the lock: check the architecture,
// raise the dynamic shared-memory limit of every kernel instantiation and
// look up the status word's device address.
int device_setup(int* dev_out, unsigned** status_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return MHA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    st.ready = true;
    st.ok = false;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      st.ready = false;
      return MHA_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MHA_ERR_NO_DEVICE;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        st.ready = false;
        return MHA_ERR_CUDA;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    bool fail = false;
    auto smem_attr = [&](auto kernel, int bytes) {
      fail |= cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
              cudaSuccess;
    };
    smem_attr(mha::mha_fwd_kernel<64, false, false>, mha::FwdCfg<64, false>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<64, true, false>, mha::FwdCfg<64, false>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, false, false>, mha::FwdCfg<128, false>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, true, false>, mha::FwdCfg<128, false>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, false, false, false, true>, mha::FwdCfg<128, false>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, true, false, false, true>, mha::FwdCfg<128, false>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<64, false, true>, mha::FwdCfg<64, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<64, true, true>, mha::FwdCfg<64, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, false, true>, mha::FwdCfg<128, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, true, true>, mha::FwdCfg<128, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<64, false, true, true>, mha::FwdCfg<64, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<64, true, true, true>, mha::FwdCfg<64, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, false, true, true>, mha::FwdCfg<128, true>::kSmemBytes);
    smem_attr(mha::mha_fwd_kernel<128, true, true, true>, mha::FwdCfg<128, true>::kSmemBytes);
    void* sym = nullptr;
    fail |= cudaGetSymbolAddress(&sym, g_status) != cudaSuccess;
    fail |= cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            st.sms <= 0;
    if (fail) {
      st.ready = false;
      return MHA_ERR_CUDA;
    }
    st.status = static_cast<unsigned*>(sym);
    st.ok = true;
  }
  if (!st.ok) return MHA_ERR_NO_DEVICE;
  *dev_out = dev;
  *status_out = st.status;
  return MHA_OK;
}

int device_sms(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_dev[dev].sms;
}

bool encode_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_paged_map(CUtensorMap* map, const void* base, int num_blocks, int H, int page_size,
                      int d, int box_rows) {
  if (d == 128) {
    // [block * heads + head][8-row group][d-half][row][64]: one box brings
    // box_rows rows with both halves, each 8-row group's two 128-byte
    // swizzle atoms side by side (the strides need not grow outward)
    cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(page_size / 8),
                          static_cast<cuuint64_t>(num_blocks) * H};
    cuuint64_t strides[4] = {256, 128, 2048, static_cast<cuuint64_t>(page_size) * 256};
    cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(box_rows / 8), 1};
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                          strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  }
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(page_size),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(num_blocks)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(page_size) * d * 2,
                           static_cast<cuuint64_t>(H) * page_size * d * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

long long wait_limit() {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_wait_limit;
}

}  // namespace mha_host

namespace {
template <int D, bool CAUSAL, bool SPLIT = false, bool PAGED = false, bool HMAJOR = false>
cudaError_t launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                   const CUtensorMap& mo, const mha::FwdParams& prm, int sms, cudaStream_t stream);

template <bool PAGED>
cudaError_t launch_split(int d, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const mha::FwdParams& prm, int sms, cudaStream_t st) {
  if (d == 64)
    return causal ? launch<64, true, true, PAGED>(mq, mk, mv, mq, prm, sms, st)
                  : launch<64, false, true, PAGED>(mq, mk, mv, mq, prm, sms, st);
  return causal ? launch<128, true, true, PAGED>(mq, mk, mv, mq, prm, sms, st)
                : launch<128, false, true, PAGED>(mq, mk, mv, mq, prm, sms, st);
}
}  // namespace

namespace mha_host {

// Zeroes the split pass's work-tile counter with a one-thread kernel; the
// split pass is launched next as its programmatic dependent.
static cudaError_t reset_counter(int* counter, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(1, 1, 1);
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, mha::split_counter_reset_kernel, counter);
}

int fwd_split_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      int* tile_counter, int BH, int Nq, int Nk, int d, float scale, bool causal,
                      int num_splits, int tiles_per_split, int dev, unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!encode_map(&mq, q, BH, Nq, d, 128) || !encode_map(&mk, k, BH, Nk, d, 128) ||
      !encode_map(&mv, v, BH, Nk, d, 128))
    return MHA_ERR_CUDA;
  mha::FwdParams prm = {};
  prm.status = status;
  prm.wait_limit = wait_limit();
  prm.N = Nk;
  prm.num_mblocks = 1;
  prm.BH = BH;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.num_splits = num_splits;
  prm.tiles_per_split = tiles_per_split;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.tile_counter = tile_counter;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (reset_counter(tile_counter, st) != cudaSuccess) return MHA_ERR_CUDA;
  const cudaError_t err = launch_split<false>(d, causal, mq, mk, mv, prm, device_sms(dev), st);
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int fwd_paged_partial(const void* q, const void* k_cache, const void* v_cache,
                      const int* block_table, const int* seq_lens, float* o_part, float* lse_part,
                      int* tile_counter, int B, int H, int Nq, int d, int page_size, int num_blocks,
                      int max_blocks, float scale, bool causal, int num_splits, int tiles_per_split, int dev,
                      unsigned* status, cudaStream_t st) {
  const int BH = B * H;
  const int rows = page_size < 128 ? page_size : 128;
  CUtensorMap mq, mk, mv;
  if (!encode_map(&mq, q, BH, Nq, d, 128) ||
      !encode_paged_map(&mk, k_cache, num_blocks, H, page_size, d, rows) ||
      !encode_paged_map(&mv, v_cache, num_blocks, H, page_size, d, rows))
    return MHA_ERR_CUDA;
  mha::FwdParams prm = {};
  prm.status = status;
  prm.wait_limit = wait_limit();
  prm.N = max_blocks * page_size;
  prm.num_mblocks = 1;
  prm.BH = BH;
  prm.Nq = Nq;
  prm.Nk = max_blocks * page_size;
  prm.num_splits = num_splits;
  prm.tiles_per_split = tiles_per_split;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.page_size = page_size;
  prm.max_blocks = max_blocks;
  prm.num_heads = H;
  prm.num_blocks = num_blocks;
  prm.tile_counter = tile_counter;
  if (reset_counter(tile_counter, st) != cudaSuccess) return MHA_ERR_CUDA;
  const cudaError_t err = launch_split<true>(d, causal, mq, mk, mv, prm, device_sms(dev), st);
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace mha_host

namespace {
using namespace mha_host;

// The head-major order (m-blocks of one head adjacent; causal: pairs of
// m-blocks of equal total cost, one pair per CTA per round) keeps the K/V of
// the few heads in flight in L2.  It is used at d = 128 once all heads' K/V
// no longer fit in L2, unless its rounds of equal work items would leave
// more than 5% of the grid idle: the other order's snake rounds balance
// unequal tiles better (at 2 x 32 heads x 4096 keys, causal, 512 pairs on
// 152 SMs fill 84% of the last round's slots and measured 4% slower).
bool use_head_major(int BH, int N, int d, bool causal, int sms) {
  const double kv_bytes = 2.0 * BH * static_cast<double>(N) * d * 2.0;
  if (d != 128 || kv_bytes <= 96.0 * (1 << 20)) return false;
  const long long mblocks = (N + 255) / 256;
  const long long items = static_cast<long long>(BH) * (causal ? (mblocks + 1) / 2 : mblocks);
  const long long grid = items < sms ? items : sms;
  const long long rounds = (items + grid - 1) / grid;
  return static_cast<double>(items) >= 0.95 * static_cast<double>(rounds * grid);
}

// Persistent launch: one CTA per SM (fewer when there are fewer work tiles),
// each walking its share of the (bh, m-block) or (bh, split) tiles.
// `mo` is used by the d = 128 square pass only (the others store O with
// plain stores); callers of the other passes pass any map there.
template <int D, bool CAUSAL, bool SPLIT, bool PAGED, bool HMAJOR>
cudaError_t launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                   const CUtensorMap& mo, const mha::FwdParams& prm, int sms, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  // work tiles, or for the head-major order work items (causal: pairs of m-blocks)
  const long long total =
      static_cast<long long>(prm.BH) *
      (SPLIT ? prm.num_splits : (HMAJOR && CAUSAL ? (prm.num_mblocks + 1) / 2 : prm.num_mblocks));
  cfg.gridDim = dim3(static_cast<unsigned>(total < sms ? total : sms), 1, 1);
  cfg.blockDim = dim3(mha::FwdCfg<D, SPLIT>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = mha::FwdCfg<D, SPLIT>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  cudaLaunchAttribute attr[1] = {};
  if (SPLIT) {
    // a programmatic dependent of split_counter_reset_kernel, queued just
    // before it (the kernel waits for that one before its first read)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  using OArg = mha::OMapArg<mha::FwdCfg<D, SPLIT>::kOSets != 0>;
  OArg oarg;
  if constexpr (mha::FwdCfg<D, SPLIT>::kOSets != 0) oarg.map = mo;
  return cudaLaunchKernelEx(&cfg, mha::mha_fwd_kernel<D, CAUSAL, SPLIT, PAGED, HMAJOR>, mq, mk, mv, oarg, prm);
}

}  // namespace

extern "C" {

const char* mha_strerror(int status) {
  switch (status) {
    case MHA_OK: return "ok";
    case MHA_ERR_INVALID_ARG: return "invalid argument";
    case MHA_ERR_UNSUPPORTED_DIM: return "unsupported head dimension (d must be 64 or 128)";
    case MHA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MHA_ERR_CUDA: return "CUDA call failed";
    case MHA_ERR_TIMEOUT: return "device-side wait timed out";
    case MHA_ERR_NO_DEVICE: return "no usable sm_103 device";
    case MHA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the built-in 16 MiB buffer";
    default: return "unknown status";
  }
}

int mha_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
            int d, float scale, int causal, void* stream) {
  if (B < 0 || H < 0 || N < 0) return MHA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return MHA_ERR_UNSUPPORTED_DIM;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MHA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || N == 0) return MHA_OK;
  if (BH > 0x7fffffffll) return MHA_ERR_INVALID_ARG;
  // the kernel counts work tiles (and their positions past the end) in int
  if (BH * ((N + 255) / 256) > (1ll << 30)) return MHA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return MHA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return MHA_ERR_MISALIGNED;
  // the outputs must not overlap the inputs
  const uintptr_t tb = static_cast<uintptr_t>(BH) * N * d * 2;
  const uintptr_t lb = static_cast<uintptr_t>(BH) * N * 4;
  for (const void* in : {q, k, v})
    if (overlap(o, tb, in, tb) || overlap(lse, lb, in, tb)) return MHA_ERR_INVALID_ARG;
  if (overlap(o, tb, lse, lb)) return MHA_ERR_INVALID_ARG;

  int dev = 0;
  unsigned* status = nullptr;
  const int rc = device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;

  // at d = 128 O is written by TMA stores of 32-row boxes (one softmax
  // warp's rows); at d = 64 the kernel stores O directly and gets the Q map
  // in the O map's place, which it never uses
  CUtensorMap mq, mk, mv, mo;
  if (!encode_map(&mq, q, static_cast<int>(BH), N, d, 128) ||
      !encode_map(&mk, k, static_cast<int>(BH), N, d, 128) ||
      !encode_map(&mv, v, static_cast<int>(BH), N, d, 128))
    return MHA_ERR_CUDA;
  if (d == 128) {
    if (!encode_map(&mo, o, static_cast<int>(BH), N, d, 32)) return MHA_ERR_CUDA;
  } else {
    mo = mq;
  }

  mha::FwdParams prm = {};
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.status = status;
  prm.wait_limit = wait_limit();
  prm.N = N;
  prm.num_mblocks = (N + 255) / 256;
  prm.BH = static_cast<int>(BH);
  const int sms = device_sms(dev);
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (d == 64)
    err = causal ? launch<64, true>(mq, mk, mv, mo, prm, sms, st)
                 : launch<64, false>(mq, mk, mv, mo, prm, sms, st);
  else if (use_head_major(static_cast<int>(BH), N, d, causal != 0, sms))
    err = causal ? launch<128, true, false, false, true>(mq, mk, mv, mo, prm, sms, st)
                 : launch<128, false, false, false, true>(mq, mk, mv, mo, prm, sms, st);
  else
    err = causal ? launch<128, true>(mq, mk, mv, mo, prm, sms, st)
                 : launch<128, false>(mq, mk, mv, mo, prm, sms, st);
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int mha_fwd_tile_order(int B, int H, int N, int d, int causal, int sms, int* order) {
  if (B < 0 || H < 0 || N < 0 || sms <= 0 || order == nullptr) return MHA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return MHA_ERR_UNSUPPORTED_DIM;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffll) return MHA_ERR_INVALID_ARG;
  if (BH * ((N + 255) / 256) > (1ll << 30)) return MHA_ERR_INVALID_ARG;  // as mha_fwd
  *order = (BH > 0 && N > 0 && use_head_major(static_cast<int>(BH), N, d, causal != 0, sms)) ? 1 : 0;
  return MHA_OK;
}

int mha_device_status(void* stream, int reset, unsigned* detail) {
  int dev = 0;
  unsigned* status = nullptr;
  const int rc = device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MHA_ERR_CUDA;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MHA_ERR_CUDA;
  if (reset && word != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MHA_ERR_CUDA;
  }
  if (detail) *detail = word;
  return (word & mha::kStatusTimeout) ? MHA_ERR_TIMEOUT : MHA_OK;
}

int mha_set_wait_limit(long long cycles) {
  if (cycles <= 0) return MHA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_wait_limit = cycles;
  return MHA_OK;
}

int mha_wait_selftest(long long cycles, void* stream) {
  if (cycles <= 0 || cycles > (1ll << 34)) return MHA_ERR_INVALID_ARG;
  int dev = 0;
  unsigned* status = nullptr;
  int rc = device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = st;
  if (cudaLaunchKernelEx(&cfg, mha::wait_selftest_kernel, status, cycles) != cudaSuccess)
    return MHA_ERR_CUDA;
  unsigned word = 0;
  rc = mha_device_status(stream, 1, &word);
  if (rc == MHA_ERR_TIMEOUT && (word & mha::kSiteSelftest) == 0) return MHA_ERR_CUDA;
  return rc;
}

}  // extern "C"
