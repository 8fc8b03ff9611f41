// Stage 4: greedy acceptance of the verified tree.
//
// "Bastion: Budget-Aware Speculative Decoding with Tree-structured Block
// Diffusion Drafting" (explainer gist.science/de/paper/2605.29727),
// "Experimentelle Ergebnisse": greedy decoding at temperature 0; the tree
// verification keeps the longest continuation the target agrees with
// ("Akzeptanzlänge").  Per tree node the target's greedy token is the argmax of
// its logits; the accepted path starts at the root and follows the child whose
// token equals its parent's greedy token.
//
// Design: one thread-block cluster per (request, node) row splits the
// vocabulary into C chunks streamed with 16-byte loads (the HBM-bound part);
// each thread keeps its first maximum, the CTA and then the cluster (through
// distributed shared memory) reduce (value desc, id asc) keys.  The row's
// cluster then takes a ticket on its request; the cluster that completes the
// request's last row walks the tree (one warp, ballots over the children) and
// returns the ticket word to zero.
#include <cooperative_groups.h>
#include <math_constants.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace bst {

constexpr int K4_THREADS = 256;
constexpr int K4_WARPS = K4_THREADS / 32;
constexpr int K4_U = 16;      // 16-byte loads per thread: 64 KB per CTA in flight
constexpr int K4_MAXC = 16;

template <class Tag, bool kVecOK>
__global__ void __launch_bounds__(K4_THREADS, 2) accept_kernel(
    const void *__restrict__ target, int n_max, int V, int64_t row_stride, int K, int chunk,
    const int32_t *__restrict__ n_g, const int32_t *__restrict__ parent, const int32_t *__restrict__ token,
    int32_t *__restrict__ acc_len, int32_t *__restrict__ acc_nodes, int32_t *__restrict__ acc_tok,
    int32_t *__restrict__ bonus, int32_t *__restrict__ argmax_out, uint32_t *__restrict__ tickets,
    int32_t *__restrict__ amax_ws, uint32_t *__restrict__ dev_err) {
  constexpr int VEC = Tag::kVec;
  constexpr int PER = K4_U * VEC;
  constexpr int TILE = K4_THREADS * PER;
  using T = typename Tag::storage;

  __shared__ uint64_t s_red[K4_WARPS];
  __shared__ uint64_t s_best;
  __shared__ int s_last;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int crank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.y;
  const int b = row / n_max;
  const int i = row - b * n_max;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nb = n_g[b];

  if (nb < 1 || nb > n_max) {   // uniform for the whole cluster
    if (i == 0 && crank == 0 && tid == 0) {
      set_err(dev_err, BASTION_DEVERR_N);
      acc_len[b] = -1;
      bonus[b] = -1;
      for (int j = 0; j <= K; ++j) acc_nodes[b * (K + 1) + j] = -1, acc_tok[b * (K + 1) + j] = -1;
    }
    if (argmax_out && i == 0 && crank == 0)
      for (int j = tid; j < n_max; j += K4_THREADS) argmax_out[static_cast<int64_t>(b) * n_max + j] = -1;
    return;
  }
  if (i >= nb) {
    if (argmax_out && crank == 0 && tid == 0) argmax_out[row] = -1;
    return;
  }

  // ---- streaming argmax over this CTA's chunk
  const T *rowp = reinterpret_cast<const T *>(target) + static_cast<int64_t>(row) * row_stride;
  const int c0 = crank * chunk;
  const int c1 = min(V, c0 + chunk);
  float bv = -CUDART_INF_F;
  int32_t bi = -1;
  for (int base = c0; base < c1; base += TILE) {
    // the tile stays packed in registers (16 bytes per load); padding
    // positions past the chunk hold -inf
    uint4 raw[K4_U];
#pragma unroll
    for (int u = 0; u < K4_U; ++u) {
      const int e0 = base + (u * K4_THREADS + tid) * VEC;
      if (kVecOK && e0 + VEC <= c1) {
        raw[u] = ld_stream16(rowp + e0);
      } else {
        float f[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) f[j] = (e0 + j < c1) ? load_scalar<Tag>(rowp, e0 + j) : -CUDART_INF_F;
        raw[u] = pack16<Tag>(f);
      }
    }
#define X(idx) elem16<Tag>(raw[(idx) / VEC], (idx) % VEC)
    float tm = -CUDART_INF_F;
#pragma unroll
    for (int u = 0; u < K4_U; ++u) tm = fmaxf(tm, vmax16<Tag>(raw[u]));
    if (tm > bv) {
      // first position (lowest id) holding the tile maximum; elements of a
      // thread are visited in increasing id order
      int32_t first = -1;
#pragma unroll
      for (int u = K4_U - 1; u >= 0; --u)
#pragma unroll
        for (int j = VEC - 1; j >= 0; --j)
          if (X(u * VEC + j) == tm) first = base + (u * K4_THREADS + tid) * VEC + j;
      bv = tm;
      bi = first;
    }
  }
  uint64_t key = (bi >= 0) ? pack_vi(bv, bi) : 0ull;
  key = warp_max_u64(key);
  if (lane == 0) s_red[tid >> 5] = key;
  __syncthreads();
  if (tid == 0) {
    uint64_t m = s_red[0];
#pragma unroll
    for (int w = 1; w < K4_WARPS; ++w) m = s_red[w] > m ? s_red[w] : m;
    s_best = m;
  }
  cluster.sync();
  if (crank == 0 && tid == 0) {
    uint64_t m = 0;
    for (int c = 0; c < C; ++c) {
      const uint64_t o = *cluster.map_shared_rank(&s_best, c);
      m = o > m ? o : m;
    }
    const int32_t a = packed_i(m);
    amax_ws[row] = a;
    if (argmax_out) argmax_out[row] = a;
    __threadfence();
    const uint32_t t = atomicAdd(&tickets[b], 1u);
    s_last = (t == static_cast<uint32_t>(nb - 1)) ? 1 : 0;
  }
  cluster.sync();   // remote shared memory no longer needed after this point
  if (crank != 0) return;
  __syncthreads();
  if (!s_last) return;

  // ---- this cluster finished the request's last row: walk the tree
  if (tid < 32) {
    __threadfence();
    const int32_t *par = parent + static_cast<int64_t>(b) * n_max;
    const int32_t *tk = token + static_cast<int64_t>(b) * n_max;
    const int32_t *am = amax_ws + static_cast<int64_t>(b) * n_max;
    int u = 0;
    int len = 0;
    int32_t a = __ldcg(am);
    if (lane == 0) acc_nodes[b * (K + 1)] = 0;
    while (len < K) {
      int found = -1;
      for (int v0 = 1; v0 < nb; v0 += 32) {
        const int v = v0 + lane;
        const bool hit = (v < nb) && (par[v] == u) && (tk[v] == a);
        const unsigned m = __ballot_sync(FULL, hit);
        if (m) {
          found = v0 + __ffs(m) - 1;
          break;
        }
      }
      if (found < 0) break;
      ++len;
      if (lane == 0) {
        acc_nodes[b * (K + 1) + len] = found;
        acc_tok[b * (K + 1) + len - 1] = a;
      }
      u = found;
      a = __ldcg(am + u);
    }
    if (lane == 0) {
      acc_len[b] = len;
      bonus[b] = a;
      acc_tok[b * (K + 1) + len] = a;
      for (int j = len + 1; j <= K; ++j) acc_nodes[b * (K + 1) + j] = -1;
      for (int j = len + 1; j <= K; ++j) acc_tok[b * (K + 1) + j] = -1;
      tickets[b] = 0u;   // the workspace word is zero again for the next call
    }
  }
}

size_t accept_workspace_size(int B, int n_max) {
  const size_t t = (static_cast<size_t>(B) * 4 + 255) / 256 * 256;
  return t + static_cast<size_t>(B) * n_max * 4;
}

cudaError_t launch_accept(const void *target, bool bf16, int B, int n_max, int V, int64_t row_stride, int K,
                          const int32_t *n, const int32_t *parent, const int32_t *token, int32_t *acc_len,
                          int32_t *acc_nodes, int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out, void *ws,
                          uint32_t *dev_err, int num_sms, cudaStream_t stream) {
  const int esz = bf16 ? 2 : 4;
  const int rows = B * n_max;
  // CTAs per row: first enough that each CTA's chunk is one tile (all of its
  // loads in flight at once), then more while the grid is under two CTAs per SM
  const int tile = K4_THREADS * K4_U * (16 / esz);
  int C = 1;
  while (C < K4_MAXC && (V + C - 1) / C > tile) C <<= 1;
  while (C < K4_MAXC && static_cast<int64_t>(rows) * C < 2LL * num_sms && V / (2 * C) >= 4096) C <<= 1;
  const int vec = 16 / esz;
  int chunk = (V + C - 1) / C;
  chunk = (chunk + vec - 1) / vec * vec;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(target) % 16 == 0) && ((row_stride * esz) % 16 == 0);
  uint32_t *tickets = reinterpret_cast<uint32_t *>(ws);
  int32_t *amax_ws = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(ws) + (static_cast<size_t>(B) * 4 + 255) / 256 * 256);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, rows, 1);
  cfg.blockDim = dim3(K4_THREADS, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define BST_ACCEPT_ARGS target, n_max, V, row_stride, K, chunk, n, parent, token, acc_len, acc_nodes, acc_tok, bonus, argmax_out, tickets, amax_ws, dev_err
  if (bf16) {
    if (vec_ok) return cudaLaunchKernelEx(&cfg, accept_kernel<BF16Tag, true>, BST_ACCEPT_ARGS);
    return cudaLaunchKernelEx(&cfg, accept_kernel<BF16Tag, false>, BST_ACCEPT_ARGS);
  }
  if (vec_ok) return cudaLaunchKernelEx(&cfg, accept_kernel<F32Tag, true>, BST_ACCEPT_ARGS);
  return cudaLaunchKernelEx(&cfg, accept_kernel<F32Tag, false>, BST_ACCEPT_ARGS);
#undef BST_ACCEPT_ARGS
}

cudaError_t prepare_accept() {
  cudaError_t e;
  e = cudaFuncSetAttribute(accept_kernel<BF16Tag, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(accept_kernel<BF16Tag, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(accept_kernel<F32Tag, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(accept_kernel<F32Tag, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace bst
