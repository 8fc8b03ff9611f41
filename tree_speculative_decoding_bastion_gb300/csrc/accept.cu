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
// Design (HBM-bound vocabulary pass): a row is cut into C chunks; CTA
// (c, b, z) takes chunk c of the rows z, z + Y, ... of request b below its tree
// size (grid stride, so a small tree in a large budget launches few idle CTAs).
// Per row it stages the chunk into shared memory with bulk asynchronous copies
// (cp.async.bulk, all of it in flight at once, the next row prefetched into
// L2), finds the chunk's first maximum and publishes it as a 64-bit key
// (value desc, id asc) with one atomicMax on the row's slot in the workspace;
// after its last row it takes one ticket on its request for all of its rows.
// The CTA that completes the request walks the tree (one warp, ballots over
// the children) and returns the row slots and the ticket to zero for the next
// call.  No clusters, no inter-CTA waiting.
#include <math_constants.h>

#include <algorithm>

#include "sm100_ptx.cuh"

namespace bst {

#ifdef BST_TRACE
__device__ unsigned long long g_k4_trace[4096 * 16];
extern "C" cudaError_t bastion_trace_read_accept(void *dst, size_t bytes) {
  return cudaMemcpyFromSymbol(dst, g_k4_trace, bytes);
}
#endif

constexpr int K4_THREADS = 256;
constexpr int K4_WARPS = K4_THREADS / 32;
constexpr int K4_MAX_CHUNK_BYTES = 48 * 1024;   // shared memory per CTA
constexpr uint64_t K4_WAIT_NS = 200ull * 1000ull * 1000ull;

// Workspace: [tickets: B x u32, padded to 256 B][row keys: B x n_max x u64]
__host__ __device__ inline size_t accept_ticket_bytes(int B) { return (static_cast<size_t>(B) * 4 + 255) / 256 * 256; }

template <class Tag, bool kBulk>
__global__ void __launch_bounds__(K4_THREADS) accept_kernel(
    const void *__restrict__ target, int n_max, int V, int64_t row_stride, int K, int chunk, int C,
    const int32_t *__restrict__ n_g, const int32_t *__restrict__ parent, const int32_t *__restrict__ token,
    int32_t *__restrict__ acc_len, int32_t *__restrict__ acc_nodes, int32_t *__restrict__ acc_tok,
    int32_t *__restrict__ bonus, int32_t *__restrict__ argmax_out, uint32_t *__restrict__ tickets,
    unsigned long long *__restrict__ rowkey, uint32_t *__restrict__ dev_err) {
  constexpr int VEC = Tag::kVec;
  using T = typename Tag::storage;
  extern __shared__ __align__(128) uint8_t k4_smem[];
  __shared__ uint64_t s_bar;
  __shared__ unsigned long long s_red[K4_WARPS];
  __shared__ int s_last;
  __shared__ int s_dead;   // a staged copy never landed: issue no further copies
  __shared__ int32_t s_am[BASTION_MAX_NODES], s_par[BASTION_MAX_NODES], s_tok[BASTION_MAX_NODES];

  // CTA (crank, b, z) takes chunk crank of the rows z, z + Y, ... of request b
  const int crank = blockIdx.x;
  const int b = blockIdx.y;
  const int z = blockIdx.z;
  const int Y = gridDim.z;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const T *req = reinterpret_cast<const T *>(target) + static_cast<int64_t>(b) * n_max * row_stride;
  const int c0 = crank * chunk;
  const int c1 = min(V, c0 + chunk);
  const int len = max(0, c1 - c0);
  if (tid == 0) BST_STAMP(g_k4_trace, 0);
  if (kBulk && tid == 0) {
    s_dead = 0;
    mbar_init(&s_bar, 1);
    fence_mbar_init();
    // warm L2 with the first chunk while the producing grid finishes
    if (len > 0 && z < n_max)
      prefetch_l2_bulk(req + static_cast<int64_t>(z) * row_stride + c0, static_cast<uint32_t>(len) * sizeof(T));
  }
  pdl_wait();
  pdl_trigger();
  if (tid == 0) BST_STAMP(g_k4_trace, 5);
  const int nb = n_g[b];

  if (nb < 1 || nb > n_max) {   // the whole request is invalid
    if (z == 0 && crank == 0 && tid == 0) {
      set_err(dev_err, BASTION_DEVERR_N);
      acc_len[b] = -1;
      bonus[b] = -1;
      for (int j = 0; j <= K; ++j) acc_nodes[b * (K + 1) + j] = -1, acc_tok[b * (K + 1) + j] = -1;
    }
    if (argmax_out && z == 0 && crank == 0)
      for (int j = tid; j < n_max; j += K4_THREADS) argmax_out[static_cast<int64_t>(b) * n_max + j] = -1;
    return;
  }
  if (z >= nb) return;   // no row of this request for this CTA

  if (kBulk) __syncthreads();   // the barrier was initialised before the dependency wait

  // the request's tree, for the walk in case this CTA completes the request
  auto stage_tree = [&]() {
    for (int j = tid; j < nb; j += K4_THREADS) {
      s_par[j] = parent[static_cast<int64_t>(b) * n_max + j];
      s_tok[j] = token[static_cast<int64_t>(b) * n_max + j];
    }
  };
  int it = 0;
  int dead_it = -1;   // the row whose staged copy timed out (kBulk)
  for (int i = z; i < nb; i += Y, ++it) {
    const int row = b * n_max + i;
    const T *rowp = req + static_cast<int64_t>(i) * row_stride;
    float bv = -CUDART_INF_F;
    int32_t bi = -1;
    if (kBulk) {
      // ---- stage the chunk into shared memory with bulk copies
      const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
      // s_dead was last written before the previous row's barrier, so every
      // thread reads the same value here
      const bool dead = s_dead != 0;
      if (tid == 0 && bytes > 0 && !dead) {
        mbar_expect_tx(&s_bar, bytes);
        for (uint32_t off = 0; off < bytes; off += 16384u) {
          const uint32_t nbytes = min(16384u, bytes - off);
          bulk_load(k4_smem + off, reinterpret_cast<const uint8_t *>(rowp + c0) + off, nbytes, &s_bar);
        }
        // and warm L2 with this CTA's next row
        if (i + Y < nb) prefetch_l2_bulk(rowp + static_cast<int64_t>(Y) * row_stride + c0, bytes);
      }
      if (it == 0) stage_tree();   // while the first chunk is in flight
      int no_abort = 0;
      if (dead) {
        // an earlier copy of this CTA never landed: the row counts as empty
        // (its ticket is still taken, so the request completes and the
        // workspace returns to zero)
      } else if (bytes > 0 && !mbar_wait(&s_bar, it & 1, &no_abort, K4_WAIT_NS)) {
        s_dead = 1;
        dead_it = it;
        set_err(dev_err, BASTION_DEVERR_TIMEOUT);
      } else {
        // thread t scans 16-byte vectors t, t + 256, ... in increasing order, so
        // a strict ">" keeps its first maximum
        const uint4 *v4 = reinterpret_cast<const uint4 *>(k4_smem);
        const int nvec = len / VEC;
        for (int v = tid; v < nvec; v += K4_THREADS) {
          const uint4 x = v4[v];
          const float m = vmax16<Tag>(x);
          if (m > bv) {
            int32_t first = -1;
#pragma unroll
            for (int j = VEC - 1; j >= 0; --j)
              if (elem16<Tag>(x, j) == m) first = c0 + v * VEC + j;
            bv = m;
            bi = first;
          }
        }
      }
    } else {
      if (it == 0) stage_tree();
      // unaligned rows: scalar loads, each thread strides over the chunk
      for (int e = c0 + tid; e < c1; e += K4_THREADS) {
        const float x = load_scalar<Tag>(rowp, e);
        if (x > bv) bv = x, bi = e;
      }
    }
    if (tid == 0) BST_STAMP(g_k4_trace, 1);
    unsigned long long key = (bi >= 0) ? pack_vi(bv, bi) : 0ull;
    key = warp_max_u64(key);
    if (lane == 0) s_red[tid >> 5] = key;
    __syncthreads();   // also: every thread is done with the staged chunk
    if (tid == 0) {
      unsigned long long m = s_red[0];
#pragma unroll
      for (int w = 1; w < K4_WARPS; ++w) m = s_red[w] > m ? s_red[w] : m;
      if (m) atomicMax(&rowkey[row], m);
      BST_STAMP(g_k4_trace, 2);
    }
    // (one barrier a row: the next row's copy is issued by thread 0 only
    // after it has read s_red, and the other warps write s_red again only
    // after that copy has landed)
  }
  // One ticket per CTA for all of its rows, (row, chunk) pairs counted:
  // release -- this CTA's row slot updates (thread 0's atomics) are visible
  // to the CTA that completes the count; acquire -- that CTA then sees every
  // other CTA's updates.  (A ticket per row made every row wait for a GPU
  // round trip: 34.5 -> 33.0 us on 4 x 128 rows of 151936.)
  if (tid == 0) {
    const uint32_t mine = static_cast<uint32_t>(it);   // rows this CTA took
    const uint32_t t = atomic_add_acq_rel_gpu(&tickets[b], mine);
    s_last = (t + mine == static_cast<uint32_t>(nb * C)) ? 1 : 0;
  }
  __syncthreads();
  if (kBulk && dead_it >= 0) {
    // let the copy that timed out land (bounded) before this CTA's shared
    // memory can go to another CTA
    int no_abort = 0;
    mbar_wait(&s_bar, dead_it & 1, &no_abort, K4_WAIT_NS);
  }
  if (!s_last) return;

  // ---- this CTA completed the request: argmax per node, then walk the tree
  // (argmax, parent and token rows in shared memory: the walk itself touches
  // no global memory)
  unsigned long long *rk = rowkey + static_cast<int64_t>(b) * n_max;
  for (int j = tid; j < n_max; j += K4_THREADS) {
    if (j < nb) {
      const int32_t am = packed_i(__ldcg(rk + j));
      s_am[j] = am;
      if (argmax_out) argmax_out[static_cast<int64_t>(b) * n_max + j] = am;
    } else if (argmax_out) {
      argmax_out[static_cast<int64_t>(b) * n_max + j] = -1;
    }
  }
  __syncthreads();
  if (tid < 32) {
    int u = 0;
    int len2 = 0;
    int32_t a = s_am[0];
    if (lane == 0) acc_nodes[b * (K + 1)] = 0;
    while (len2 < K) {
      // children come after their parent in the best-first order
      int found = -1;
      for (int v0 = u + 1; v0 < nb; v0 += 32) {
        const int v = v0 + lane;
        const bool hit = (v < nb) && (s_par[v] == u) && (s_tok[v] == a);
        const unsigned m = __ballot_sync(FULL, hit);
        if (m) {
          found = v0 + __ffs(m) - 1;
          break;
        }
      }
      if (found < 0) break;
      ++len2;
      if (lane == 0) {
        acc_nodes[b * (K + 1) + len2] = found;
        acc_tok[b * (K + 1) + len2 - 1] = a;
      }
      u = found;
      a = s_am[u];
    }
    if (lane == 0) {
      acc_len[b] = len2;
      bonus[b] = a;
      acc_tok[b * (K + 1) + len2] = a;
      for (int j = len2 + 1; j <= K; ++j) acc_nodes[b * (K + 1) + j] = -1;
      for (int j = len2 + 1; j <= K; ++j) acc_tok[b * (K + 1) + j] = -1;
      BST_STAMP(g_k4_trace, 3);
    }
  }
  __syncthreads();
  // the workspace words are zero again for the next call
  for (int j = tid; j < nb; j += K4_THREADS) rk[j] = 0ull;
  if (tid == 0) tickets[b] = 0u;
}

size_t accept_workspace_size(int B, int n_max) {
  return accept_ticket_bytes(B) + static_cast<size_t>(B) * n_max * 8;
}

cudaError_t launch_accept(const void *target, bool bf16, int B, int n_max, int V, int64_t row_stride, int K,
                          const int32_t *n, const int32_t *parent, const int32_t *token, int32_t *acc_len,
                          int32_t *acc_nodes, int32_t *acc_tok, int32_t *bonus, int32_t *argmax_out, void *ws,
                          uint32_t *dev_err, int num_sms, cudaStream_t stream) {
  const int esz = bf16 ? 2 : 4;
  const int vec = 16 / esz;
  // CTAs per row: chunks of at most 48 KB, each a multiple of 16 bytes
  const int max_chunk = K4_MAX_CHUNK_BYTES / esz;
  int C = (V + max_chunk - 1) / max_chunk;
  int chunk = (V + C - 1) / C;
  chunk = (chunk + vec - 1) / vec * vec;
  C = (V + chunk - 1) / chunk;
  const bool bulk = (reinterpret_cast<uintptr_t>(target) % 16 == 0) && ((row_stride * esz) % 16 == 0) &&
                    ((static_cast<int64_t>(V) * esz) % 16 == 0);
  uint32_t *tickets = reinterpret_cast<uint32_t *>(ws);
  auto *rowkey = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(ws) + accept_ticket_bytes(B));
  // rows per request handled by Y CTAs each (grid stride): enough CTAs for
  // about two waves at four per SM, never more than one per row; the tree's
  // size is a device value, so the grid covers n_max rows
  const int64_t want = (8LL * num_sms + static_cast<int64_t>(C) * B - 1) / (static_cast<int64_t>(C) * B);
  const int Y = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(n_max, want)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, B, Y);
  cfg.blockDim = dim3(K4_THREADS, 1, 1);
  cfg.dynamicSmemBytes = bulk ? static_cast<size_t>(chunk) * esz : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = fill_launch_attrs(attr);
#define BST_ACCEPT_ARGS target, n_max, V, row_stride, K, chunk, C, n, parent, token, acc_len, acc_nodes, acc_tok, \
                        bonus, argmax_out, tickets, rowkey, dev_err
  if (bf16) {
    if (bulk) return cudaLaunchKernelEx(&cfg, accept_kernel<BF16Tag, true>, BST_ACCEPT_ARGS);
    return cudaLaunchKernelEx(&cfg, accept_kernel<BF16Tag, false>, BST_ACCEPT_ARGS);
  }
  if (bulk) return cudaLaunchKernelEx(&cfg, accept_kernel<F32Tag, true>, BST_ACCEPT_ARGS);
  return cudaLaunchKernelEx(&cfg, accept_kernel<F32Tag, false>, BST_ACCEPT_ARGS);
#undef BST_ACCEPT_ARGS
}

cudaError_t prepare_accept() {
  cudaError_t e;
  e = cudaFuncSetAttribute(accept_kernel<BF16Tag, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, K4_MAX_CHUNK_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(accept_kernel<F32Tag, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, K4_MAX_CHUNK_BYTES);
  if (e != cudaSuccess) return e;
  if ((e = prefer_max_shared(accept_kernel<BF16Tag, true>)) != cudaSuccess) return e;
  if ((e = prefer_max_shared(accept_kernel<BF16Tag, false>)) != cudaSuccess) return e;
  if ((e = prefer_max_shared(accept_kernel<F32Tag, true>)) != cudaSuccess) return e;
  return prefer_max_shared(accept_kernel<F32Tag, false>);
}

}  // namespace bst
