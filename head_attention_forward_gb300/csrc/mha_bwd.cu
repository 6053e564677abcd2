// mha_bwd.cu - host side of the attention backward: argument checks, tensor
// maps, launches, and the extern "C" entry points mha_bwd and
// mha_bwd_workspace_size that include/mha_fwd.h declares.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "mha_bwd_kernel.cuh"
#include "mha_fwd.h"
#include "mha_internal.h"

namespace {
using namespace mha_host;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_attr_done[kMaxDevices] = {};

template <int D, bool CAUSAL, bool DKDV>
bool set_smem_attr() {
  return cudaFuncSetAttribute(mha::bwd_tile_kernel<D, CAUSAL, DKDV>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              mha::BwdCfg<D>::kSmemBytes) == cudaSuccess;
}

// Raise the shared-memory limit of every tile-kernel instantiation, once per
// device.
int ensure_attrs(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_attr_done[dev]) return MHA_OK;
  bool ok = set_smem_attr<64, false, false>() && set_smem_attr<64, false, true>() &&
            set_smem_attr<64, true, false>() && set_smem_attr<64, true, true>() &&
            set_smem_attr<128, false, false>() && set_smem_attr<128, false, true>() &&
            set_smem_attr<128, true, false>() && set_smem_attr<128, true, true>();
  if (!ok) return MHA_ERR_CUDA;
  g_attr_done[dev] = true;
  return MHA_OK;
}

size_t dsum_bytes(long long BH, int N) {
  return (static_cast<size_t>(BH) * static_cast<size_t>(N) * 4 + 15) & ~static_cast<size_t>(15);
}

template <int D, bool CAUSAL, bool DKDV>
cudaError_t launch_tile(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mdo, const mha::BwdParams& prm, int BH,
                        cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = prm.tiles_fastest
                    ? dim3(static_cast<unsigned>(prm.n_tiles), static_cast<unsigned>(BH), 1)
                    : dim3(static_cast<unsigned>(BH), static_cast<unsigned>(prm.n_tiles), 1);
  cfg.blockDim = dim3(mha::BwdCfg<D>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = mha::BwdCfg<D>::kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, mha::bwd_tile_kernel<D, CAUSAL, DKDV>, mq, mk, mv, mdo, prm);
}

template <int D>
cudaError_t launch_all(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mdo, const mha::BwdParams& prm, const void* o,
                       const void* dout, float* dsum, long long BH, int N, bool causal,
                       cudaStream_t st) {
  const long long rows = BH * N;
  constexpr int kRows = mha::RowdotCfg<D>::kRowsPerBlock;
  mha::bwd_rowdot_kernel<D><<<static_cast<unsigned>((rows + kRows - 1) / kRows), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), dsum, rows);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int bh = static_cast<int>(BH);
  if (causal) {
    err = launch_tile<D, true, true>(mq, mk, mv, mdo, prm, bh, st);
    if (err == cudaSuccess) err = launch_tile<D, true, false>(mq, mk, mv, mdo, prm, bh, st);
  } else {
    err = launch_tile<D, false, true>(mq, mk, mv, mdo, prm, bh, st);
    if (err == cudaSuccess) err = launch_tile<D, false, false>(mq, mk, mv, mdo, prm, bh, st);
  }
  return err;
}

}  // namespace

extern "C" {

size_t mha_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || (d != 64 && d != 128)) return 0;
  return dsum_bytes(static_cast<long long>(B) * H, N);
}

int mha_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
            const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
            float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || N < 0) return MHA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return MHA_ERR_UNSUPPORTED_DIM;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MHA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || N == 0) return MHA_OK;
  if (BH > 0x7fffffffll) return MHA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return MHA_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, o, static_cast<const void*>(lse), dout,
                          static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv), static_cast<const void*>(workspace)})
    if (!aligned16(ptr)) return MHA_ERR_MISALIGNED;
  const size_t need = dsum_bytes(BH, N);
  if (workspace_bytes < need) return MHA_ERR_INVALID_ARG;
  // outputs and workspace overlap nothing else
  const size_t tb = static_cast<size_t>(BH) * N * d * 2;
  const size_t lb = static_cast<size_t>(BH) * N * 4;
  struct Span { const void* p; size_t n; };
  const Span ins[] = {{q, tb}, {k, tb}, {v, tb}, {o, tb}, {lse, lb}, {dout, tb}};
  const Span outs[] = {{dq, tb}, {dk, tb}, {dv, tb}, {workspace, need}};
  for (int a = 0; a < 4; ++a) {
    for (const Span& in : ins)
      if (overlap(outs[a].p, outs[a].n, in.p, in.n)) return MHA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlap(outs[a].p, outs[a].n, outs[b].p, outs[b].n)) return MHA_ERR_INVALID_ARG;
  }

  int dev = 0;
  unsigned* status = nullptr;
  int rc = device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;
  rc = ensure_attrs(dev);
  if (rc != MHA_OK) return rc;

  CUtensorMap mq, mk, mv, mdo;
  const int bh = static_cast<int>(BH);
  if (!encode_map(&mq, q, bh, N, d, 128) || !encode_map(&mk, k, bh, N, d, 128) ||
      !encode_map(&mv, v, bh, N, d, 128) || !encode_map(&mdo, dout, bh, N, d, 128))
    return MHA_ERR_CUDA;

  float* dsum = static_cast<float*>(workspace);
  mha::BwdParams prm = {};
  prm.lse = lse;
  prm.dsum = dsum;
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.status = status;
  prm.wait_limit = wait_limit();
  prm.N = N;
  prm.n_tiles = (N + 127) / 128;
  // 32+ tiles per head: one head's CTAs together (measured +5..8% at N >= 4096,
  // -10% at N = 2048 causal); grid y is limited to 65535
  prm.tiles_fastest = (prm.n_tiles >= 32 && BH <= 65535) ? 1 : 0;
  prm.scale = scale;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err =
      d == 64 ? launch_all<64>(mq, mk, mv, mdo, prm, o, dout, dsum, BH, N, causal != 0, st)
              : launch_all<128>(mq, mk, mv, mdo, prm, o, dout, dsum, BH, N, causal != 0, st);
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"
