// After acceptance: the accepted path's keys and values join the context cache.
//
// FlexDraft page ("FlexDraft: Flexible Speculative Decoding via Attention
// Tuning and Bonus-Guided Calibration"), "Flex-Decoding", decoupled execution:
// once the accepted length is known, drafting continues from the verified
// prefix and reuses the KV cache of the target's verification pass.  BASTION
// ("Bastion: Budget-Aware Speculative Decoding with Tree-structured Block
// Diffusion Drafting"), "Das Ergebnis": every step's accepted tokens extend the
// text.  In this library's reading the tree's root (node 0, the token the
// previous step emitted, at position ctx_len) and the a accepted draft tokens
// were all keyed by the verification pass, so request b appends the a + 1 rows
// k_tree[b, acc_nodes[b, j], h, :] (j = 0..a, root first) at context
// positions ctx_len[b] + j of every KV head h, and its context grows to
// ctx_len[b] + a + 1; the bonus token is the next step's root.
//
// Design: pure data movement of (a + 1) * Hkv rows of d elements for K and V
// per request (at most 33 * Hkv * d * 2 elements, tens of KB), so one CTA per
// request copies its rows with 16-byte vectors; the element type does not
// matter.  All checks (acc_len, node ids, capacity, page ids) are made before
// the copy by the threads that own them and combined with one barrier, so a
// bad request copies nothing.  That barrier also separates every read of
// ctx_len[b] from the write of ctx_out[b], which may therefore alias it.
#include "common.cuh"

namespace bst {

constexpr int KC_THREADS = 256;

__global__ void __launch_bounds__(KC_THREADS) kv_commit_kernel(
    const uint4 *__restrict__ k_tree, const uint4 *__restrict__ v_tree, int n_max, int Hkv, int row_vecs, int K,
    const int32_t *__restrict__ acc_len, const int32_t *__restrict__ acc_nodes, uint4 *kc, uint4 *vc,
    int64_t L_max, const int32_t *__restrict__ block_table, int max_pages, int num_pages, int page_size,
    const int32_t *ctx_len, int32_t *ctx_out, uint32_t *__restrict__ dev_err) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const bool paged = block_table != nullptr;
  pdl_wait();   // the accepted path comes from the previous stage
  const int a = acc_len[b];
  const int c = ctx_len[b];
  // request-level checks, one thread per path entry
  uint32_t bad = 0;
  if (a < 0 || a > K) {
    bad = BASTION_DEVERR_N;
  } else if (c < 0 || (paged ? (static_cast<int64_t>(c) + a) / page_size >= max_pages
                             : static_cast<int64_t>(c) + a >= L_max)) {
    bad = BASTION_DEVERR_CTX;
  } else if (tid <= a) {
    const int node = acc_nodes[static_cast<int64_t>(b) * (K + 1) + tid];
    if (node < 0 || node >= n_max) bad = BASTION_DEVERR_N;
    if (paged) {
      const int p = c + tid;
      const int page = block_table[static_cast<int64_t>(b) * max_pages + p / page_size];
      if (page < 0 || page >= num_pages) bad |= BASTION_DEVERR_PAGE;
    }
  }
  if (bad && (tid == 0 || tid <= a)) set_err(dev_err, bad);
  const bool ok = !__syncthreads_or(bad != 0);   // also: every read of ctx_len[b] is done
  pdl_trigger();
  if (ok) {
    const int per_kv = (a + 1) * Hkv * row_vecs;   // vectors of K (then as many of V)
    for (int t = tid; t < 2 * per_kv; t += KC_THREADS) {
      const int is_v = t >= per_kv;
      const int u = is_v ? t - per_kv : t;
      const int vi = u % row_vecs;
      const int r = u / row_vecs;
      const int h = r % Hkv;
      const int j = r / Hkv;
      const int node = acc_nodes[static_cast<int64_t>(b) * (K + 1) + j];
      const int p = c + j;
      const int64_t src = ((static_cast<int64_t>(b) * n_max + node) * Hkv + h) * row_vecs + vi;
      int64_t dst;
      if (paged) {
        const int page = block_table[static_cast<int64_t>(b) * max_pages + p / page_size];
        dst = ((static_cast<int64_t>(page) * Hkv + h) * page_size + p % page_size) * row_vecs + vi;
      } else {
        dst = ((static_cast<int64_t>(b) * Hkv + h) * L_max + p) * row_vecs + vi;
      }
      if (is_v)
        vc[dst] = __ldg(v_tree + src);
      else
        kc[dst] = __ldg(k_tree + src);
    }
  }
  if (tid == 0) ctx_out[b] = ok ? c + a + 1 : c;
}

cudaError_t launch_kv_commit(const void *k_tree, const void *v_tree, int esz, int B, int n_max, int Hkv, int d, int K,
                             const int32_t *acc_len, const int32_t *acc_nodes, void *kc, void *vc, int64_t L_max,
                             const int32_t *block_table, int max_pages, int num_pages, int page_size,
                             const int32_t *ctx_len, int32_t *ctx_out, uint32_t *dev_err, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, 1, 1);
  cfg.blockDim = dim3(KC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = fill_launch_attrs(attr);
  const int row_vecs = d * esz / 16;
  return cudaLaunchKernelEx(&cfg, kv_commit_kernel, static_cast<const uint4 *>(k_tree),
                            static_cast<const uint4 *>(v_tree), n_max, Hkv, row_vecs, K, acc_len, acc_nodes,
                            static_cast<uint4 *>(kc), static_cast<uint4 *>(vc), L_max, block_table, max_pages,
                            num_pages, page_size, ctx_len, ctx_out, dev_err);
}

}  // namespace bst
