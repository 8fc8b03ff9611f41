// Stage 2: best-first prefix tree with the online budget stop.
//
// "Bastion: Budget-Aware Speculative Decoding with Tree-structured Block
// Diffusion Drafting" (explainer gist.science/de/paper/2605.29727), Methodik:
//   §1 "Pfad-Bewertung": node i at depth d(i) scores rho(i) = prod_{k=1}^{d(i)} q_k(x_ik);
//      "Randverteilungs-Unabhängigkeit": the candidates of each position combine
//      freely, so a depth-d node offers the top-k tokens of position d+1;
//   §2 A_hat(T) = sum_{i in T} rho(i); best-first repeatedly adds the valid node
//      with the highest rho;
//   §3 the controller grows the tree until S(N) = A_hat(T_N) L_AR / C(N) starts
//      to fall.
//
// Design: one CTA per request.  Because the children of a node are the same
// sorted top-k list for every parent at that depth, each tree node keeps only
// its best not-yet-added child as its frontier candidate ("next child"
// pointer); the frontier then has at most one entry per node.  Warp 0 owns the
// frontier: node i lives in lane i % 32, register slot i / 32, as a 64-bit key
// (sortable fp32 log-rho | token | parent) so that one pair of warp max
// reductions (redux.sync) yields the next node with the exact tie-break
// (rho desc, token asc, parent asc).  The candidate table is packed as
// {logit, token word} pairs, the lse prefix as {hi, lo} float pairs and the
// node state as {path sum, depth | next rank}, so a pop reads everything it
// needs with five 64-bit shared loads.  Every lane computes the two new keys
// (the parent's next child, the new node's best child), the owning lanes take
// them with predicated moves, and every lane writes the same node state, so
// the loop has no divergent branch and no warp barrier.  With the controller
// the pops run until the stop rule can first apply (n_min + 1 nodes) and then
// in chunks of 8; after each chunk the lanes evaluate rho, A_hat and the
// S(n+1) < S(n) test in parallel and the first drop ends the tree.  The
// confidence threshold (FlexDraft page, "Flex-Decoding", selective
// verification) is a second stop test in the same place: past n_min, a node
// whose fp32 log rho is below log tau ends the tree.
// Arithmetic is fp32 except single float64 additions for the lse prefix
// (this GPU's FP64 pipe is narrow, so no float64 exp/log/division).
#include <math_constants.h>

#include "common.cuh"

namespace bst {

#ifdef BST_TRACE
__device__ unsigned long long g_k2_trace[4096 * 16];
extern "C" cudaError_t bastion_trace_read_tree(void *dst, size_t bytes) {
  return cudaMemcpyFromSymbol(dst, g_k2_trace, bytes);
}
#endif

constexpr int K2_THREADS = 256;

struct K2Smem {
  uint2 E[BASTION_MAX_DEPTH * BASTION_MAX_TOPK];   // [K][k]: {logit bits, (0x3FFFF - token) << 8}
  double P64[BASTION_MAX_DEPTH + 1];   // sum of lse over positions 1..d
  float2 PP[BASTION_MAX_DEPTH + 2];    // P64 as a float pair (hi, lo); one spare entry
  uint2 NS[BASTION_MAX_NODES];         // {fp32 logit sum of the path (bits), depth | next rank << 8}
  int2 PT[BASTION_MAX_NODES];          // {parent, token}
  float rho[BASTION_MAX_NODES];
  float ahat[BASTION_MAX_NODES];       // ahat[j] = A_hat after nodes 0..j
  int n_final;
};

// Frontier key of a candidate with path sum S, table entry e = {logit, token
// word} at key depth d (PP[d]) and parent byte parb = 255 - parent: high word
// sortable fp32 log rho (rho desc), low word (0x3FFFF - token) << 8 | parb.
BST_DEV uint64_t cand_key2(float S, float2 pp, uint32_t tokw, uint32_t parb) {
  const float key = (S - pp.x) - pp.y;   // log rho, fp32
  return (static_cast<uint64_t>(sortable(key)) << 32) | tokw | parb;
}

template <int SLOTS>
__global__ void __launch_bounds__(K2_THREADS) tree_build_kernel(
    const int32_t *__restrict__ ids_g, const float *__restrict__ lg_g, const double *__restrict__ lse_g,
    int K, int k, int V, const int32_t *__restrict__ root_tok, const int32_t *__restrict__ ctx_len,
    int n_min, int n_max, const float *__restrict__ Ctab, float L_AR, float log_tau, int32_t *__restrict__ n_out,
    int32_t *__restrict__ parent, int32_t *__restrict__ token, int32_t *__restrict__ depth,
    int32_t *__restrict__ pos, float *__restrict__ rho_out, unsigned long long *__restrict__ mask,
    float *__restrict__ ahat_out, float *__restrict__ S_out, float *__restrict__ S_curve,
    uint32_t *__restrict__ dev_err) {
  __shared__ K2Smem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const bool controller = (Ctab != nullptr);
  const bool tau_on = log_tau > -CUDART_INF_F;   // confidence threshold (log tau, fp32)
  const bool eval = controller || tau_on;         // the tree size is decided by a stop rule

  if (tid == 0) BST_STAMP(g_k2_trace, 0);
  pdl_wait();
  pdl_trigger();
  if (tid == 0) BST_STAMP(g_k2_trace, 4);
  // ---- load the request's candidate table
  for (int e = tid; e < K * k; e += K2_THREADS) {
    int32_t id = ids_g[static_cast<int64_t>(b) * K * k + e];
    if (id < 0 || id >= V) {
      set_err(dev_err, BASTION_DEVERR_TOKEN);
      id = 0;
    }
    sm.E[e] = make_uint2(__float_as_uint(lg_g[static_cast<int64_t>(b) * K * k + e]),
                         (0x3FFFFu - static_cast<uint32_t>(id)) << 8);
  }
  if (tid < 32) {
    // prefix of the positions' lse (warp scan; K <= 32), kept in float64 and as
    // an fp32 pair hi + lo for the fp32 keys of the serial loop
    double P = (tid < K) ? lse_g[static_cast<int64_t>(b) * K + tid] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(FULL, P, o);
      if (tid >= o) P += y;
    }
    if (tid < K) {
      sm.P64[tid + 1] = P;
      const float hi = static_cast<float>(P);
      sm.PP[tid + 1] = make_float2(hi, static_cast<float>(P - static_cast<double>(hi)));
    }
  }
  if (tid == 0) {
    sm.P64[0] = 0.0;
    sm.PP[0] = make_float2(0.f, 0.f);
    sm.PP[K + 1] = make_float2(0.f, 0.f);
    int32_t rt = root_tok[b];
    if (rt < 0 || rt >= V) set_err(dev_err, BASTION_DEVERR_TOKEN);
    sm.PT[0] = make_int2(-1, rt);
    sm.NS[0] = make_uint2(__float_as_uint(0.f), 0u);
    sm.rho[0] = 1.f;
    sm.ahat[0] = 1.f;
    sm.n_final = 1;
  }
  __syncthreads();

  if (tid == 0) BST_STAMP(g_k2_trace, 1);
  // ---- warp 0: best-first expansion.  Every lane runs the same instruction
  // stream: both new frontier keys are computed by all lanes, and the two
  // owning lanes take them with predicated moves.
  if (tid < 32) {
    uint64_t slot[SLOTS];
#pragma unroll
    for (int r = 0; r < SLOTS; ++r) slot[r] = 0ull;
    if (lane == 0) slot[0] = cand_key2(__uint_as_float(sm.E[0].x), sm.PP[1], sm.E[0].y, 255u);
    uint64_t best = slot[0];

    int n = 1;
    int n_final = -1;
    int chunk_start = 1;
    while (n_final < 0) {
      // with a stop rule, pop until it can first apply (n_min + 1 nodes),
      // then test it every 8 pops
      const int target = eval ? min(n_max, max(n + 8, n_min + 1)) : n_max;
      bool exhausted = false;
      while (n < target) {
        const uint32_t bh = static_cast<uint32_t>(best >> 32);
        const uint32_t mh = __reduce_max_sync(FULL, bh);
        if (mh == 0u) {
          exhausted = true;
          break;
        }
        const uint32_t ml = __reduce_max_sync(FULL, bh == mh ? static_cast<uint32_t>(best) : 0u);
        const int p = 255 - static_cast<int>(ml & 0xFFu);
        const int tokn = 0x3FFFF - static_cast<int>(ml >> 8);
        const int t = n;
        const uint2 ns = sm.NS[p];
        const float Sp = __uint_as_float(ns.x);
        const int dcp = static_cast<int>(ns.y);
        const int dp = dcp & 0xFF;
        const int c = dcp >> 8;
        const int dt = dp + 1;
        const int base = dp * k + c;
        const bool vP = c + 1 < k;    // node p has a next child
        const bool vT = dt < K;       // the new node has children
        const uint2 e0 = sm.E[base];                  // the popped candidate
        const uint2 e1 = sm.E[vP ? base + 1 : 0];     // p's next child
        const uint2 f0 = sm.E[vT ? dt * k : 0];       // t's best child
        const float2 pp1 = sm.PP[dt];
        const float2 pp2 = sm.PP[dt + 1];
        const float St = Sp + __uint_as_float(e0.x);   // the same sum the popped key was made from
        const uint64_t kP = vP ? cand_key2(Sp + __uint_as_float(e1.x), pp1, e1.y, 255u - static_cast<uint32_t>(p)) : 0ull;
        const uint64_t kT = vT ? cand_key2(St + __uint_as_float(f0.x), pp2, f0.y, 255u - static_cast<uint32_t>(t)) : 0ull;
        // every lane stores the same values (no divergent branch); each lane
        // then reads back its own writes, so the loop needs no warp barrier
        sm.NS[t] = make_uint2(__float_as_uint(St), static_cast<uint32_t>(dt));
        sm.NS[p].y = static_cast<uint32_t>(dcp + 256);
        sm.PT[t] = make_int2(p, tokn);
        best = 0ull;
#pragma unroll
        for (int r = 0; r < SLOTS; ++r) {
          const int me = r * 32 + lane;
          slot[r] = (me == p) ? kP : slot[r];
          slot[r] = (me == t) ? kT : slot[r];
          best = slot[r] > best ? slot[r] : best;
        }
        ++n;
      }
      __syncwarp();
      if (eval) {
        // rho, A_hat and the stop tests for the nodes of this chunk, 32 at a time
        for (int cs = chunk_start; cs < n && n_final < 0; cs += 32) {
          const int j = cs + lane;
          float r = 0.f;
          float key = 0.f;
          if (j < n) {
            const uint2 nj = sm.NS[j];
            key = static_cast<float>(static_cast<double>(__uint_as_float(nj.x)) - sm.P64[nj.y & 0xFF]);
            r = expf(key);
            sm.rho[j] = r;
          }
          // inclusive prefix sum over the lanes
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(FULL, r, o);
            if (lane >= o) r += y;
          }
          const float base = sm.ahat[cs - 1];
          const float a_next = base + r;                  // A_hat(j + 1)
          float a_prev = __shfl_up_sync(FULL, a_next, 1);
          if (lane == 0) a_prev = base;                   // A_hat(j)
          if (j < n) sm.ahat[j] = a_next;
          // tree of size j grows to j + 1 only if S(j + 1) >= S(j) and node
          // j's rho (the cumulative draft confidence of its path) is >= tau
          // (short-circuit order: C is read only for j < n <= n_max)
          const bool drop = (j < n) && (j >= n_min) &&
                            ((controller && a_next * Ctab[j] < a_prev * Ctab[j + 1]) || (tau_on && key < log_tau));
          const unsigned dm = __ballot_sync(FULL, drop);
          if (dm) n_final = cs + (__ffs(dm) - 1);
          __syncwarp();
        }
        if (n_final < 0 && (exhausted || n >= n_max)) n_final = n;
        chunk_start = n;
      } else {
        n_final = n;
      }
    }
    if (lane == 0) sm.n_final = n_final;
    if (lane == 0) BST_STAMP(g_k2_trace, 2);
  }
  __syncthreads();
  const int nf = sm.n_final;

  // ---- rho and A_hat for a fixed budget (a stop rule filled them already)
  if (!eval) {
    for (int j = 1 + tid; j < nf; j += K2_THREADS) {
      const uint2 nj = sm.NS[j];
      const float key = static_cast<float>(static_cast<double>(__uint_as_float(nj.x)) - sm.P64[nj.y & 0xFF]);
      sm.rho[j] = expf(key);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l sums nodes [8l, 8l+8), then an exclusive scan over lanes
      float part = 0.f;
      for (int j = 8 * lane; j < min(8 * lane + 8, nf); ++j) part += sm.rho[j];
      float incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      float run = incl - part;
      for (int j = 8 * lane; j < min(8 * lane + 8, nf); ++j) {
        run += sm.rho[j];
        sm.ahat[j] = run;
      }
    }
    __syncthreads();
  }

  // ---- outputs
  const int W = (n_max + 63) >> 6;
  const int64_t row0 = static_cast<int64_t>(b) * n_max;
  const int cl = ctx_len[b];
  for (int i = tid; i < n_max; i += K2_THREADS) {
    const int64_t o = row0 + i;
    if (i < nf) {
      const int2 pt = sm.PT[i];
      const int di = static_cast<int>(sm.NS[i].y & 0xFFu);
      parent[o] = pt.x;
      token[o] = pt.y;
      depth[o] = di;
      pos[o] = cl + di;
      rho_out[o] = sm.rho[i];
      if (S_curve) {
        const float c = controller ? Ctab[i + 1] : 1.f;
        S_curve[o] = sm.ahat[i] * L_AR / c;
      }
      unsigned long long m0 = 0, m1 = 0, m2 = 0, m3 = 0;
      int j = i;
      while (j >= 0) {
        const unsigned long long bit = 1ull << (j & 63);
        const int w = j >> 6;
        if (w == 0) m0 |= bit;
        else if (w == 1) m1 |= bit;
        else if (w == 2) m2 |= bit;
        else m3 |= bit;
        j = sm.PT[j].x;
      }
      unsigned long long *mrow = mask + o * W;
      mrow[0] = m0;
      if (W > 1) mrow[1] = m1;
      if (W > 2) mrow[2] = m2;
      if (W > 3) mrow[3] = m3;
    } else {
      parent[o] = -1;
      token[o] = -1;
      depth[o] = -1;
      pos[o] = -1;
      rho_out[o] = 0.f;
      if (S_curve) S_curve[o] = 0.f;
      unsigned long long *mrow = mask + o * W;
      for (int w = 0; w < W; ++w) mrow[w] = 0ull;
    }
  }
  if (tid == 0) BST_STAMP(g_k2_trace, 3);
  if (tid == 0) {
    n_out[b] = nf;
    const float a = sm.ahat[nf - 1];
    const float c = controller ? Ctab[nf] : 1.f;
    ahat_out[b] = a;
    S_out[b] = a * L_AR / c;
  }
}

cudaError_t launch_tree_build(const int32_t *ids, const float *lg, const double *lse, int B, int K, int k,
                              int V, const int32_t *root_tok, const int32_t *ctx_len, int n_min, int n_max,
                              const float *C, float L_AR, float log_tau, int32_t *n, int32_t *parent,
                              int32_t *token, int32_t *depth, int32_t *pos, float *rho, uint64_t *mask, float *ahat,
                              float *S, float *S_curve, uint32_t *dev_err, cudaStream_t stream) {
  auto *m = reinterpret_cast<unsigned long long *>(mask);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, 1, 1);
  cfg.blockDim = dim3(K2_THREADS, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = fill_launch_attrs(attr);
  // frontier slots per lane: one per 32 nodes of the budget
  auto *fn = n_max <= 64 ? tree_build_kernel<2> : n_max <= 128 ? tree_build_kernel<4> : tree_build_kernel<8>;
  return cudaLaunchKernelEx(&cfg, fn, ids, lg, lse, K, k, V, root_tok, ctx_len, n_min, n_max, C, L_AR, log_tau, n, parent,
                            token, depth, pos, rho, m, ahat, S, S_curve, dev_err);
}

cudaError_t prepare_tree_build() {
  cudaError_t e;
  if ((e = prefer_max_shared(tree_build_kernel<2>)) != cudaSuccess) return e;
  if ((e = prefer_max_shared(tree_build_kernel<4>)) != cudaSuccess) return e;
  return prefer_max_shared(tree_build_kernel<8>);
}

}  // namespace bst
