// bastion_accept_noalloc: greedy acceptance for callers that cannot allocate.
//
// bastion_accept needs a caller-allocated workspace (one ticket word per
// request and one argmax slot per tree node).  Some callers have no way to
// allocate it: engines that hand all free GPU memory to the KV cache at start-up
// and keep no allocator reachable from the decode step, or code that must not
// take the implicit device synchronisation a cudaMalloc/cudaFree can cause.
// This variant keeps that scratch in a fixed array in this library's device
// memory instead.  Inputs and outputs are still the caller's.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/bastion.h"

namespace bst {
void set_last_error(const std::string &msg);
size_t accept_workspace_size(int B, int n_max);
cudaError_t launch_accept(const void *target, bool bf16, int B, int n_max, int V, int64_t row_stride, int K,
                          const int32_t *n, const int32_t *parent, const int32_t *token, int32_t *acc_len,
                          int32_t *acc_nodes, int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out, void *ws,
                          uint32_t *dev_err, int num_sms, cudaStream_t stream);
}  // namespace bst

// The scratch every call of bastion_accept_noalloc uses: ticket words first,
// then the per-node argmax.  Every GPU that loads this library holds these
// bytes until the process exits.
static __device__ __align__(256) unsigned char g_accept_scratch[BASTION_ACCEPT_NOALLOC_MAX_BYTES];

namespace {

constexpr int kMaxDevices = 64;
struct ScratchState {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  void *ptr = nullptr;   // device address of g_accept_scratch on that device
  int sms = 0;
};
ScratchState g_scratch[kMaxDevices];

// the explanation goes where bastion_last_error() reads it
bastion_status noalloc_fail(bastion_status s, const std::string &m) {
  bst::set_last_error(m);
  return s;
}

}  // namespace

namespace bst {
// Set-up of `dev`, once per device, with `dev` current (bastion_init runs it
// while it prepares the device, so the first library call on a device does
// it): the host-side name of the array is not a device address, so look the
// address up.  A failure is kept and reported by bastion_accept_noalloc.
void prepare_accept_noalloc(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return;
  ScratchState &st = g_scratch[dev];
  std::call_once(st.once, [&] {
    st.err = cudaGetSymbolAddress(&st.ptr, g_accept_scratch);
    cudaDeviceProp prop;
    if (st.err == cudaSuccess) st.err = cudaGetDeviceProperties(&prop, dev);
    if (st.err == cudaSuccess) st.sms = prop.multiProcessorCount;
  });
}
}  // namespace bst

extern "C" bastion_status bastion_accept_noalloc(const void *target, bastion_dtype dtype, int B, int n_max, int V,
                                                 int64_t row_stride, int K, const int32_t *n,
                                                 const int32_t *parent, const int32_t *token, int32_t *acc_len,
                                                 int32_t *acc_nodes, int32_t *acc_tok, int32_t *bonus,
                                                 int32_t *argmax_out, uint32_t *dev_err, bastion_stream_t stream) {
  if (!target || !n || !parent || !token || !acc_len || !acc_nodes || !acc_tok || !bonus)
    return noalloc_fail(BASTION_ERR_INVALID_ARG, "accept_noalloc: NULL pointer");
  if (dtype != BASTION_F32 && dtype != BASTION_BF16)
    return noalloc_fail(BASTION_ERR_INVALID_ARG, "accept_noalloc: bad dtype");
  if (B < 1 || n_max < 1 || V < 1 || K < 1 || row_stride < V)
    return noalloc_fail(BASTION_ERR_INVALID_ARG, "accept_noalloc: bad sizes");
  if (V > BASTION_MAX_VOCAB || K > BASTION_MAX_DEPTH || n_max > BASTION_MAX_NODES ||
      static_cast<int64_t>(B) * n_max > 65535)
    return noalloc_fail(BASTION_ERR_UNSUPPORTED, "accept_noalloc: V <= 262144, K <= 32, n_max <= 256, B*n_max <= 65535");
  const size_t need = bst::accept_workspace_size(B, n_max);
  if (need > sizeof(g_accept_scratch))
    return noalloc_fail(BASTION_ERR_UNSUPPORTED,
                        "accept_noalloc: needs " + std::to_string(need) + " bytes of scratch, the built-in array has " +
                            std::to_string(sizeof(g_accept_scratch)) + " (use bastion_accept with a workspace)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(BASTION_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(BASTION_ERR_NO_DEVICE, "accept_noalloc: device index too large");
  // bastion_init prepares the device, the scratch address included
  bastion_status s = bastion_init(dev);
  if (s != BASTION_OK) return s;   // bastion_init already recorded why
  ScratchState &st = g_scratch[dev];
  bst::prepare_accept_noalloc(dev);   // no-op once done
  if (st.err != cudaSuccess || !st.ptr)
    return noalloc_fail(BASTION_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(st.err));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // the ticket words and row slots must start at zero; clear them on the
  // caller's stream
  e = cudaMemsetAsync(st.ptr, 0, need, cs);
  if (e != cudaSuccess) return noalloc_fail(BASTION_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  e = bst::launch_accept(target, dtype == BASTION_BF16, B, n_max, V, row_stride, K, n, parent, token, acc_len,
                         acc_nodes, acc_tok, bonus, argmax_out, st.ptr, dev_err, st.sms, cs);
  if (e != cudaSuccess) return noalloc_fail(BASTION_ERR_CUDA, std::string("accept_noalloc launch: ") + cudaGetErrorString(e));
  return BASTION_OK;
}
