// C ABI of the spec-tree step: argument checks, per-device set-up, TMA tensor
// maps and kernel launches.  Nothing here allocates device memory or waits on
// a stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/bastion.h"

namespace bst {
cudaError_t prepare_topk_softmax();
cudaError_t prepare_accept();
cudaError_t prepare_tree_attn();
cudaError_t prepare_tree_build();
cudaError_t launch_topk_softmax(const void *logits, bool bf16, int rows, int V, int64_t row_stride, int k,
                                int32_t *ids, float *lg, float *q, double *lse, uint32_t *dev_err, int num_sms,
                                cudaStream_t stream);
cudaError_t launch_tree_build(const int32_t *ids, const float *lg, const double *lse, int B, int K, int k, int V,
                              const int32_t *root_tok, const int32_t *ctx_len, int n_min, int n_max, const float *C,
                              float L_AR, float log_tau, int32_t *n, int32_t *parent, int32_t *token, int32_t *depth,
                              int32_t *pos, float *rho, uint64_t *mask, float *ahat, float *S, float *S_curve,
                              uint32_t *dev_err, cudaStream_t stream);
size_t accept_workspace_size(int B, int n_max);
cudaError_t launch_accept(const void *target, bool bf16, int B, int n_max, int V, int64_t row_stride, int K,
                          const int32_t *n, const int32_t *parent, const int32_t *token, int32_t *acc_len,
                          int32_t *acc_nodes, int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out, void *ws,
                          uint32_t *dev_err, int num_sms, cudaStream_t stream);
struct AttnPlan {
  int paged, mtiles, splits, nctas;
  int64_t cap;
  size_t ws_bytes, ticket_bytes;
};
AttnPlan plan_tree_attn(int B, int n_max, int Hq, int Hkv, int d, int64_t cap, int num_sms, bool paged);
cudaError_t launch_tree_attn_tc(const CUtensorMap *maps, const AttnPlan &pl, int B, int n_max, int Hq, int Hkv, int d,
                                float scale, int page_size, int max_pages, int num_pages, const int32_t *ctx_len,
                                const int32_t *n, const uint64_t *mask, const int32_t *block_table, void *out,
                                void *ws, uint32_t *dev_err, cudaStream_t stream);
cudaError_t launch_tree_attn_f32(const float *q, const float *kt, const float *vt, const float *kc, const float *vc,
                                 float *out, int B, int n_max, int Hq, int Hkv, int d, float scale, bool paged,
                                 int64_t L_max, int page_size, int max_pages, int num_pages, int64_t cap,
                                 const int32_t *ctx_len, const int32_t *n, const uint64_t *mask,
                                 const int32_t *block_table, uint32_t *dev_err, cudaStream_t stream);
cudaError_t launch_kv_commit(const void *k_tree, const void *v_tree, int esz, int B, int n_max, int Hkv, int d, int K,
                             const int32_t *acc_len, const int32_t *acc_nodes, void *kc, void *vc, int64_t L_max,
                             const int32_t *block_table, int max_pages, int num_pages, int page_size,
                             const int32_t *ctx_len, int32_t *ctx_out, uint32_t *dev_err, cudaStream_t stream);
cudaError_t launch_block_mask(int B, int n_max, int block, const int32_t *n, uint64_t *mask, uint32_t *dev_err,
                              cudaStream_t stream);
void prepare_accept_noalloc(int dev);
}  // namespace bst

namespace {

thread_local std::string g_last;

bastion_status fail(bastion_status s, const std::string &msg) {
  g_last = msg;
  return s;
}

bastion_status cuda_fail(cudaError_t e, const char *what) {
  return fail(BASTION_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
struct DeviceState {
  std::once_flag once;
  bastion_status status = BASTION_ERR_NO_DEVICE;
  std::string why;
  int sms = 0;
};
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void init_device(int device, DeviceState &st) {
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) {
    st.status = BASTION_ERR_NO_DEVICE;
    st.why = std::string("cudaGetDeviceProperties: ") + cudaGetErrorString(e);
    return;
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    st.status = BASTION_ERR_NO_DEVICE;
    st.why = "device " + std::to_string(device) + " is sm_" + std::to_string(prop.major) + std::to_string(prop.minor) +
             "; this library is built for sm_103a only";
    return;
  }
  st.sms = prop.multiProcessorCount;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  cudaError_t e1 = bst::prepare_topk_softmax();
  cudaError_t e2 = bst::prepare_accept();
  cudaError_t e3 = bst::prepare_tree_attn();
  cudaError_t e4 = bst::prepare_tree_build();
  bst::prepare_accept_noalloc(device);   // the built-in acceptance scratch's address on this device
  if (prev >= 0) cudaSetDevice(prev);
  const cudaError_t ea = e1 != cudaSuccess ? e1 : e2 != cudaSuccess ? e2 : e3 != cudaSuccess ? e3 : e4;
  if (ea != cudaSuccess) {
    st.status = BASTION_ERR_CUDA;
    st.why = std::string("setting kernel attributes failed: ") + cudaGetErrorString(ea);
    return;
  }
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    st.status = BASTION_ERR_CUDA;
    st.why = "cuTensorMapEncodeTiled is not available from the driver";
    return;
  }
  st.status = BASTION_OK;
}

// Ensures the current device is initialised; returns its SM count.
bastion_status current_device(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  bastion_status s = bastion_init(dev);
  if (s != BASTION_OK) return s;
  *sms = g_dev[dev].sms;
  return BASTION_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool encode_bf16(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                 const cuuint32_t *box) {
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int64_t kv_capacity(const bastion_kv_cache *kv) {
  return kv->block_table ? static_cast<int64_t>(kv->max_pages) * kv->page_size : kv->L_max;
}

}  // namespace

namespace bst {
// lets the other translation units of the library record an explanation
void set_last_error(const std::string &msg) { g_last = msg; }
}  // namespace bst

extern "C" {

int bastion_abi_version(void) { return 102; }

const char *bastion_status_string(bastion_status s) {
  switch (s) {
    case BASTION_OK: return "BASTION_OK";
    case BASTION_ERR_INVALID_ARG: return "BASTION_ERR_INVALID_ARG";
    case BASTION_ERR_UNSUPPORTED: return "BASTION_ERR_UNSUPPORTED";
    case BASTION_ERR_WORKSPACE: return "BASTION_ERR_WORKSPACE";
    case BASTION_ERR_CUDA: return "BASTION_ERR_CUDA";
    case BASTION_ERR_NO_DEVICE: return "BASTION_ERR_NO_DEVICE";
    case BASTION_ERR_DEVICE: return "BASTION_ERR_DEVICE";
    case BASTION_ERR_TIMEOUT: return "BASTION_ERR_TIMEOUT";
  }
  return "BASTION_ERR_UNKNOWN";
}

const char *bastion_status_str(bastion_status s) { return bastion_status_string(s); }

bastion_status bastion_read_error(const uint32_t *dev_err, uint32_t *host_word, bastion_stream_t stream) {
  if (!dev_err || !host_word) return fail(BASTION_ERR_INVALID_ARG, "read_error: NULL pointer");
  cudaError_t e = cudaMemcpyAsync(host_word, dev_err, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "read_error copy");
  return BASTION_OK;
}

bastion_status bastion_error_status(uint32_t word) {
  if (word == 0u) return BASTION_OK;
  if (word & BASTION_DEVERR_TIMEOUT) return fail(BASTION_ERR_TIMEOUT, "device error word: an in-kernel wait expired");
  return fail(BASTION_ERR_DEVICE, "device error word: bad data (bits " + std::to_string(word) + ")");
}

size_t bastion_topk_softmax_workspace_size(int rows, int V, int k) {
  (void)rows;
  (void)V;
  (void)k;
  return 0;
}

const char *bastion_last_error(void) { return g_last.c_str(); }

bastion_status bastion_init(int device) {
  if (device < 0 || device >= kMaxDevices) return fail(BASTION_ERR_INVALID_ARG, "device index out of range");
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess || device >= count)
    return fail(BASTION_ERR_NO_DEVICE, e != cudaSuccess ? std::string("cudaGetDeviceCount: ") + cudaGetErrorString(e)
                                                        : "no such CUDA device");
  DeviceState &st = g_dev[device];
  std::call_once(st.once, [&] { init_device(device, st); });
  if (st.status != BASTION_OK) return fail(st.status, st.why);
  return BASTION_OK;
}

bastion_status bastion_topk_softmax(const void *logits, bastion_dtype dtype, int rows, int V, int64_t row_stride, int k,
                                    int32_t *ids, float *lg, float *q, double *lse, uint32_t *dev_err,
                                    bastion_stream_t stream) {
  if (!logits || !ids || !lg || !q || !lse) return fail(BASTION_ERR_INVALID_ARG, "topk_softmax: NULL pointer");
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return fail(BASTION_ERR_INVALID_ARG, "topk_softmax: bad dtype");
  if (rows < 1 || V < 1 || k < 1 || row_stride < V) return fail(BASTION_ERR_INVALID_ARG, "topk_softmax: bad sizes");
  if (k > BASTION_MAX_TOPK || k > V) return fail(BASTION_ERR_UNSUPPORTED, "topk_softmax: k must be <= min(V, 32)");
  if (V > BASTION_MAX_VOCAB) return fail(BASTION_ERR_UNSUPPORTED, "topk_softmax: V > 262144");
  if (rows > 65535) return fail(BASTION_ERR_UNSUPPORTED, "topk_softmax: more than 65535 rows");
  int sms = 0;
  bastion_status s = current_device(&sms);
  if (s != BASTION_OK) return s;
  cudaError_t e = bst::launch_topk_softmax(logits, dtype == BASTION_BF16, rows, V, row_stride, k, ids, lg, q, lse,
                                           dev_err, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "topk_softmax launch");
  return BASTION_OK;
}

// shared by the two tree-build entry points (tau = 0: no threshold)
static bastion_status tree_build_impl(const int32_t *ids, const float *lg, const double *lse, int B, int K, int k, int V,
                               const int32_t *root_tok, const int32_t *ctx_len, int n_min, int n_max, const float *C,
                               float L_AR, float tau, int32_t *n, int32_t *parent, int32_t *token, int32_t *depth,
                               int32_t *pos, float *rho, uint64_t *mask, float *ahat, float *S, float *S_curve,
                               uint32_t *dev_err, bastion_stream_t stream) {
  if (!ids || !lg || !lse || !root_tok || !ctx_len || !n || !parent || !token || !depth || !pos || !rho || !mask ||
      !ahat || !S)
    return fail(BASTION_ERR_INVALID_ARG, "tree_build: NULL pointer");
  if (B < 1 || K < 1 || k < 1 || V < 1 || n_max < 1 || n_min < 1 || n_min > n_max)
    return fail(BASTION_ERR_INVALID_ARG, "tree_build: bad sizes");
  if (!(L_AR > 0.f) || !std::isfinite(L_AR)) return fail(BASTION_ERR_INVALID_ARG, "tree_build: L_AR must be > 0");
  if (!(tau >= 0.f && tau <= 1.f)) return fail(BASTION_ERR_INVALID_ARG, "tree_build: tau must lie in [0, 1]");
  if (K > BASTION_MAX_DEPTH || k > BASTION_MAX_TOPK || n_max > BASTION_MAX_NODES || V > BASTION_MAX_VOCAB)
    return fail(BASTION_ERR_UNSUPPORTED, "tree_build: K <= 32, k <= 32, n_max <= 256, V <= 262144");
  int sms = 0;
  bastion_status s = current_device(&sms);
  if (s != BASTION_OK) return s;
  // log tau in float64, rounded once to the kernel's fp32 comparison precision
  const float log_tau = tau > 0.f ? static_cast<float>(std::log(static_cast<double>(tau))) : -INFINITY;
  cudaError_t e = bst::launch_tree_build(ids, lg, lse, B, K, k, V, root_tok, ctx_len, n_min, n_max, C, L_AR, log_tau,
                                         n, parent, token, depth, pos, rho, mask, ahat, S, S_curve, dev_err,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tree_build launch");
  return BASTION_OK;
}

bastion_status bastion_tree_build(const int32_t *ids, const float *lg, const double *lse, int B, int K, int k, int V,
                                  const int32_t *root_tok, const int32_t *ctx_len, int n_min, int n_max,
                                  const float *C, float L_AR, int32_t *n, int32_t *parent, int32_t *token,
                                  int32_t *depth, int32_t *pos, float *rho, uint64_t *mask, float *ahat, float *S,
                                  float *S_curve, uint32_t *dev_err, bastion_stream_t stream) {
  return tree_build_impl(ids, lg, lse, B, K, k, V, root_tok, ctx_len, n_min, n_max, C, L_AR, 0.f, n, parent, token,
                         depth, pos, rho, mask, ahat, S, S_curve, dev_err, stream);
}

bastion_status bastion_tree_build_threshold(const int32_t *ids, const float *lg, const double *lse, int B, int K,
                                            int k, int V, const int32_t *root_tok, const int32_t *ctx_len, int n_min,
                                            int n_max, const float *C, float L_AR, float tau, int32_t *n,
                                            int32_t *parent, int32_t *token, int32_t *depth, int32_t *pos, float *rho,
                                            uint64_t *mask, float *ahat, float *S, float *S_curve, uint32_t *dev_err,
                                            bastion_stream_t stream) {
  return tree_build_impl(ids, lg, lse, B, K, k, V, root_tok, ctx_len, n_min, n_max, C, L_AR, tau, n, parent, token,
                         depth, pos, rho, mask, ahat, S, S_curve, dev_err, stream);
}

size_t bastion_tree_attn_workspace_size(int B, int n_max, int Hq, int Hkv, int d, const bastion_kv_cache *kv) {
  if (!kv || B < 1 || n_max < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (d != 64 && d != 128)) return 0;
  int sms = 0;
  if (current_device(&sms) != BASTION_OK) return 0;
  return bst::plan_tree_attn(B, n_max, Hq, Hkv, d, kv_capacity(kv), sms, kv->block_table != nullptr).ws_bytes;
}

bastion_status bastion_tree_attn(const void *q, const void *k_tree, const void *v_tree, bastion_dtype dtype, int B,
                                 int n_max, int Hq, int Hkv, int d, float scale, const bastion_kv_cache *kv,
                                 const int32_t *ctx_len, const uint64_t *mask, const int32_t *n, void *out, void *ws,
                                 size_t ws_bytes, uint32_t *dev_err, bastion_stream_t stream) {
  if (!q || !k_tree || !v_tree || !kv || !kv->k || !kv->v || !ctx_len || !mask || !n || !out)
    return fail(BASTION_ERR_INVALID_ARG, "tree_attn: NULL pointer");
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return fail(BASTION_ERR_INVALID_ARG, "tree_attn: bad dtype");
  if (B < 1 || n_max < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return fail(BASTION_ERR_INVALID_ARG, "tree_attn: bad sizes");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(BASTION_ERR_INVALID_ARG, "tree_attn: scale must be > 0");
  if (d != 64 && d != 128) return fail(BASTION_ERR_UNSUPPORTED, "tree_attn: head_dim must be 64 or 128");
  if (n_max > BASTION_MAX_NODES) return fail(BASTION_ERR_UNSUPPORTED, "tree_attn: n_max > 256");
  const bool paged = kv->block_table != nullptr;
  if (paged) {
    if (kv->max_pages < 1 || kv->num_pages < 1) return fail(BASTION_ERR_INVALID_ARG, "tree_attn: bad page counts");
    if (kv->page_size < 8 || kv->page_size > 128 || (128 % kv->page_size) != 0)
      return fail(BASTION_ERR_UNSUPPORTED, "tree_attn: page_size must be 8, 16, 32, 64 or 128");
  } else if (kv->L_max < 1) {
    return fail(BASTION_ERR_INVALID_ARG, "tree_attn: L_max must be >= 1");
  }
  const int64_t cap = kv_capacity(kv);
  if (cap > (1LL << 30)) return fail(BASTION_ERR_UNSUPPORTED, "tree_attn: context capacity too large");
  int sms = 0;
  bastion_status s = current_device(&sms);
  if (s != BASTION_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  if (dtype == BASTION_F32) {
    cudaError_t e = bst::launch_tree_attn_f32(
        static_cast<const float *>(q), static_cast<const float *>(k_tree), static_cast<const float *>(v_tree),
        static_cast<const float *>(kv->k), static_cast<const float *>(kv->v), static_cast<float *>(out), B, n_max, Hq,
        Hkv, d, scale, paged, kv->L_max, kv->page_size, kv->max_pages, kv->num_pages, cap, ctx_len, n, mask,
        kv->block_table, dev_err, st);
    if (e != cudaSuccess) return cuda_fail(e, "tree_attn (f32) launch");
    return BASTION_OK;
  }

  const int g = Hq / Hkv;
  if (g > 128 || (128 % g) != 0) return fail(BASTION_ERR_UNSUPPORTED, "tree_attn: Hq/Hkv must divide 128");
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(kv->k) || !aligned16(kv->v) ||
      !aligned16(out))
    return fail(BASTION_ERR_INVALID_ARG, "tree_attn: bf16 tensors must be 16-byte aligned");
  if (paged && B > 512) return fail(BASTION_ERR_UNSUPPORTED, "tree_attn: at most 512 requests per call (bf16, paged)");
  const bst::AttnPlan pl = bst::plan_tree_attn(B, n_max, Hq, Hkv, d, cap, sms, paged);
  if (pl.ws_bytes > 0 && (!ws || ws_bytes < pl.ws_bytes || !aligned16(ws)))
    return fail(BASTION_ERR_WORKSPACE, "tree_attn: workspace too small (need " + std::to_string(pl.ws_bytes) + " bytes)");

  CUtensorMap maps[5];
  const cuuint64_t es = 2;
  {  // Q [B*n_max][Hq][d]: box 64 x g x (128/g)
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hq),
                                static_cast<cuuint64_t>(B) * n_max};
    const cuuint64_t strides[2] = {d * es, static_cast<cuuint64_t>(Hq) * d * es};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(128 / g)};
    if (!encode_bf16(&maps[0], q, 3, dims, strides, box)) return fail(BASTION_ERR_CUDA, "tree_attn: Q tensor map");
  }
  if (!paged) {  // K/V [B*Hkv][L_max][d]: box 64 x 128 x 1
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(kv->L_max),
                                static_cast<cuuint64_t>(B) * Hkv};
    const cuuint64_t strides[2] = {d * es, static_cast<cuuint64_t>(kv->L_max) * d * es};
    const cuuint32_t box[3] = {64, 128, 1};
    if (!encode_bf16(&maps[1], kv->k, 3, dims, strides, box) || !encode_bf16(&maps[2], kv->v, 3, dims, strides, box))
      return fail(BASTION_ERR_CUDA, "tree_attn: KV tensor map");
  } else {  // pages [num_pages][Hkv][page_size][d]: box 64 x page_size x 1 x 1
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(kv->page_size),
                                static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(kv->num_pages)};
    const cuuint64_t strides[3] = {d * es, static_cast<cuuint64_t>(kv->page_size) * d * es,
                                   static_cast<cuuint64_t>(Hkv) * kv->page_size * d * es};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kv->page_size), 1, 1};
    if (!encode_bf16(&maps[1], kv->k, 4, dims, strides, box) || !encode_bf16(&maps[2], kv->v, 4, dims, strides, box))
      return fail(BASTION_ERR_CUDA, "tree_attn: paged KV tensor map");
  }
  {  // tree K/V [B*n_max][Hkv][d]: box 64 x 1 x 128
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(B) * n_max};
    const cuuint64_t strides[2] = {d * es, static_cast<cuuint64_t>(Hkv) * d * es};
    const cuuint32_t box[3] = {64, 1, 128};
    if (!encode_bf16(&maps[3], k_tree, 3, dims, strides, box) || !encode_bf16(&maps[4], v_tree, 3, dims, strides, box))
      return fail(BASTION_ERR_CUDA, "tree_attn: tree KV tensor map");
  }
  cudaError_t e = bst::launch_tree_attn_tc(maps, pl, B, n_max, Hq, Hkv, d, scale, kv->page_size, kv->max_pages,
                                           kv->num_pages, ctx_len, n, mask, kv->block_table, out, ws, dev_err, st);
  if (e != cudaSuccess) return cuda_fail(e, "tree_attn launch");
  return BASTION_OK;
}

size_t bastion_accept_workspace_size(int B, int n_max) {
  if (B < 1 || n_max < 1) return 0;
  return bst::accept_workspace_size(B, n_max);
}

bastion_status bastion_accept(const void *target, bastion_dtype dtype, int B, int n_max, int V, int64_t row_stride,
                              int K, const int32_t *n, const int32_t *parent, const int32_t *token, int32_t *acc_len,
                              int32_t *acc_nodes, int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out, void *ws,
                              size_t ws_bytes, uint32_t *dev_err, bastion_stream_t stream) {
  if (!target || !n || !parent || !token || !acc_len || !acc_nodes || !acc_tok || !bonus || !ws)
    return fail(BASTION_ERR_INVALID_ARG, "accept: NULL pointer");
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return fail(BASTION_ERR_INVALID_ARG, "accept: bad dtype");
  if (B < 1 || n_max < 1 || V < 1 || K < 1 || row_stride < V) return fail(BASTION_ERR_INVALID_ARG, "accept: bad sizes");
  if (V > BASTION_MAX_VOCAB || K > BASTION_MAX_DEPTH || n_max > BASTION_MAX_NODES)
    return fail(BASTION_ERR_UNSUPPORTED, "accept: V <= 262144, K <= 32, n_max <= 256");
  if (static_cast<int64_t>(B) * n_max > 65535) return fail(BASTION_ERR_UNSUPPORTED, "accept: B * n_max > 65535");
  if (ws_bytes < bst::accept_workspace_size(B, n_max)) return fail(BASTION_ERR_WORKSPACE, "accept: workspace too small");
  int sms = 0;
  bastion_status s = current_device(&sms);
  if (s != BASTION_OK) return s;
  cudaError_t e = bst::launch_accept(target, dtype == BASTION_BF16, B, n_max, V, row_stride, K, n, parent, token,
                                     acc_len, acc_nodes, acc_tok, bonus, argmax_out, ws, dev_err, sms,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "accept launch");
  return BASTION_OK;
}

bastion_status bastion_kv_commit(const void *k_tree, const void *v_tree, bastion_dtype dtype, int B, int n_max, int Hkv,
                                 int d, int K, const int32_t *acc_len, const int32_t *acc_nodes,
                                 const bastion_kv_cache *kv, const int32_t *ctx_len, int32_t *ctx_out,
                                 uint32_t *dev_err, bastion_stream_t stream) {
  if (!k_tree || !v_tree || !acc_len || !acc_nodes || !kv || !kv->k || !kv->v || !ctx_len || !ctx_out)
    return fail(BASTION_ERR_INVALID_ARG, "kv_commit: NULL pointer");
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return fail(BASTION_ERR_INVALID_ARG, "kv_commit: bad dtype");
  if (B < 1 || n_max < 1 || Hkv < 1 || d < 1 || K < 1) return fail(BASTION_ERR_INVALID_ARG, "kv_commit: bad sizes");
  if (n_max > BASTION_MAX_NODES || K > BASTION_MAX_DEPTH || d > 512 || B > 65535)
    return fail(BASTION_ERR_UNSUPPORTED, "kv_commit: n_max <= 256, K <= 32, d <= 512, B <= 65535");
  const int esz = dtype == BASTION_BF16 ? 2 : 4;
  if ((d * esz) % 16 != 0) return fail(BASTION_ERR_UNSUPPORTED, "kv_commit: a row of d elements must be a multiple of 16 bytes");
  if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(kv->k) || !aligned16(kv->v))
    return fail(BASTION_ERR_INVALID_ARG, "kv_commit: tensors must be 16-byte aligned");
  const bool paged = kv->block_table != nullptr;
  if (paged) {
    if (kv->max_pages < 1 || kv->num_pages < 1 || kv->page_size < 1)
      return fail(BASTION_ERR_INVALID_ARG, "kv_commit: bad page counts");
  } else if (kv->L_max < 1) {
    return fail(BASTION_ERR_INVALID_ARG, "kv_commit: L_max must be >= 1");
  }
  int sms = 0;
  bastion_status s = current_device(&sms);
  if (s != BASTION_OK) return s;
  // the cache is written: the struct's const qualifies the attention call's view
  cudaError_t e = bst::launch_kv_commit(k_tree, v_tree, esz, B, n_max, Hkv, d, K, acc_len, acc_nodes,
                                        const_cast<void *>(kv->k), const_cast<void *>(kv->v), kv->L_max,
                                        kv->block_table, kv->max_pages, kv->num_pages, kv->page_size, ctx_len,
                                        ctx_out, dev_err, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_commit launch");
  return BASTION_OK;
}

bastion_status bastion_block_mask(int B, int n_max, int block, const int32_t *n, uint64_t *mask, uint32_t *dev_err,
                                  bastion_stream_t stream) {
  if (!n || !mask) return fail(BASTION_ERR_INVALID_ARG, "block_mask: NULL pointer");
  if (B < 1 || n_max < 1 || block < 1) return fail(BASTION_ERR_INVALID_ARG, "block_mask: bad sizes");
  if (n_max > BASTION_MAX_NODES || B > 65535) return fail(BASTION_ERR_UNSUPPORTED, "block_mask: n_max <= 256, B <= 65535");
  int sms = 0;
  bastion_status s = current_device(&sms);
  if (s != BASTION_OK) return s;
  cudaError_t e = bst::launch_block_mask(B, n_max, block, n, mask, dev_err, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block_mask launch");
  return BASTION_OK;
}

}  // extern "C"
