// Stage 1: per-position marginals q_k and their top-k.
//
// "Bastion: Budget-Aware Speculative Decoding with Tree-structured Block
// Diffusion Drafting" (explainer gist.science/de/paper/2605.29727), Methodik §1:
// the block-diffusion drafter yields per-position marginals q_k(.) in a single
// forward pass; the path scores of the tree are built from these drafter
// logits.  Here q_k = softmax(logits) over the whole vocabulary and the tree
// needs only the top-k tokens of each position plus the log-normaliser.
//
// Design (HBM-bound vocabulary pass):
//   * one thread-block cluster per drafter row; the C CTAs of a cluster split
//     the vocabulary into C contiguous chunks, every byte is read once with
//     16-byte streaming loads (8 bf16 or 4 fp32 per load, U loads in flight per
//     thread);
//   * per tile the chunk lives in registers and is read twice: pass A finds the
//     maxima, pass B sums exp(x - max) and keeps candidates above a threshold
//     that provably lies below the tile's k-th largest value (a per-warp sort of
//     the lane maxima); about 2k candidates survive and are ranked exactly;
//   * the C partial results (max, sum, sorted top-k) meet in CTA rank 0 through
//     distributed shared memory, which writes ids, logits, q and lse (float64
//     output; the arithmetic is fp32 with a range-reduced logarithm).
#include <cooperative_groups.h>
#include <math_constants.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace bst {

constexpr int K1_THREADS = 256;
constexpr int K1_WARPS = K1_THREADS / 32;
constexpr int K1_U = 8;        // 16-byte loads per thread per tile
constexpr int K1_CAP = 1024;   // candidate buffer per tile
constexpr int K1_MAXC = 16;    // CTAs per cluster (row)

struct K1Smem {
  float wmax[K1_WARPS];
  float wa[K1_WARPS];          // per warp: ceil(k/8)-th largest lane maximum
  float wb[K1_WARPS];          // per warp: k-th largest lane maximum
  float wsum[K1_WARPS];
  int cnt;
  int run_n;                   // entries in the running top-k list
  float run_m;                 // running maximum of the chunk
  float run_s;                 // running sum of exp(x - run_m)
  float run_v[BASTION_MAX_TOPK];
  int32_t run_i[BASTION_MAX_TOPK];
  float new_v[BASTION_MAX_TOPK];
  int32_t new_i[BASTION_MAX_TOPK];
  float cand_v[K1_CAP + K1_MAXC * BASTION_MAX_TOPK];
  int32_t cand_i[K1_CAP + K1_MAXC * BASTION_MAX_TOPK];
  uint64_t red[K1_WARPS];
  float thr;
};

// Bitonic sort of one value per lane, descending (lane 0 gets the largest).
BST_DEV float warp_sort_desc(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      float o = __shfl_xor_sync(FULL, v, stride);
      bool up = ((lane & size) == 0);       // this block sorts descending
      bool lower = ((lane & stride) == 0);  // I hold the lower index of the pair
      // descending block: lower index keeps the max
      bool keep_max = (lower == up);
      v = keep_max ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

// Rank-select: from the M candidates in sm.cand_*, write the best min(k, M) in
// order into sm.new_* (value desc, index asc).  All threads participate.
BST_DEV void rank_select(K1Smem &sm, int M, int k) {
  for (int c = threadIdx.x; c < M; c += K1_THREADS) {
    const float v = sm.cand_v[c];
    const int32_t i = sm.cand_i[c];
    int rank = 0;
    for (int o = 0; o < M; ++o) rank += better(sm.cand_v[o], sm.cand_i[o], v, i) ? 1 : 0;
    if (rank < k) {
      sm.new_v[rank] = v;
      sm.new_i[rank] = i;
    }
  }
}

// CTA-wide maximum of a 64-bit key (all threads get it).
BST_DEV uint64_t cta_max_u64(K1Smem &sm, uint64_t x) {
  x = warp_max_u64(x);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red[w] = x;
  __syncthreads();
  uint64_t r = sm.red[0];
#pragma unroll
  for (int j = 1; j < K1_WARPS; ++j) r = sm.red[j] > r ? sm.red[j] : r;
  return r;
}

template <class Tag, bool kVecOK>
__global__ void __launch_bounds__(K1_THREADS, 2) topk_softmax_kernel(
    const void *__restrict__ logits, int V, int64_t row_stride, int k, int chunk,
    int32_t *__restrict__ ids, float *__restrict__ lg, float *__restrict__ q, double *__restrict__ lse) {
  constexpr int VEC = Tag::kVec;
  constexpr int PER = K1_U * VEC;             // elements per thread per tile
  constexpr int TILE = K1_THREADS * PER;
  using T = typename Tag::storage;

  __shared__ K1Smem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int crank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const T *rowp = reinterpret_cast<const T *>(logits) + static_cast<int64_t>(row) * row_stride;
  const int c0 = crank * chunk;
  const int c1 = min(V, c0 + chunk);
  const int kk = (k + K1_WARPS - 1) / K1_WARPS;

  if (tid == 0) {
    sm.run_n = 0;
    sm.run_m = -CUDART_INF_F;
    sm.run_s = 0.f;
    sm.cnt = 0;
  }
  __syncthreads();

  for (int base = c0; base < c1; base += TILE) {
    // the tile stays packed in registers (16 bytes per load); padding
    // positions past the chunk hold -inf
    uint4 raw[K1_U];
#pragma unroll
    for (int u = 0; u < K1_U; ++u) {
      const int e0 = base + (u * K1_THREADS + tid) * VEC;
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
    // ---- pass A: maxima and the candidate threshold
    float tm = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < PER; ++j) tm = fmaxf(tm, X(j));
    const float sorted = warp_sort_desc(tm);
    const float a_w = __shfl_sync(FULL, sorted, kk - 1);
    const float b_w = __shfl_sync(FULL, sorted, k - 1);
    if (lane == 0) {
      sm.wmax[warp] = sorted;  // lane 0 holds the warp maximum
      sm.wa[warp] = a_w;
      sm.wb[warp] = b_w;
    }
    __syncthreads();
    float mt = sm.wmax[0], amin = sm.wa[0], bmax = sm.wb[0];
#pragma unroll
    for (int w = 1; w < K1_WARPS; ++w) {
      mt = fmaxf(mt, sm.wmax[w]);
      amin = fminf(amin, sm.wa[w]);
      bmax = fmaxf(bmax, sm.wb[w]);
    }
    // Each warp has ceil(k/8) lane maxima >= its a_w, so >= k elements of the
    // tile are >= min_w a_w; likewise >= k elements are >= any single b_w.
    // Elements below the running k-th entry cannot enter the list either.
    float thr = fmaxf(amin, bmax);
    if (sm.run_n == k) thr = fmaxf(thr, sm.run_v[k - 1]);
    // ---- pass B: exp-sum and candidates
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < K1_U; ++u) {
      float sv = 0.f;
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const float xv = X(u * VEC + j);
        sv += exp2f((xv - mt) * kLog2e);   // exp(x - m); 0 for padding
        if (xv >= thr && xv > -CUDART_INF_F) {
          const int slot = atomicAdd(&sm.cnt, 1);
          if (slot < K1_CAP) {
            sm.cand_v[slot] = xv;
            sm.cand_i[slot] = base + (u * K1_THREADS + tid) * VEC + j;
          }
        }
      }
      s += sv;
    }
    s = warp_sum_f(s);
    if (lane == 0) sm.wsum[warp] = s;
    __syncthreads();
    const int cnt = sm.cnt;
    if (cnt <= K1_CAP) {
      // merge the running list into the candidate pool and rank-select
      const int rn = sm.run_n;
      for (int j = tid; j < rn; j += K1_THREADS) {
        sm.cand_v[cnt + j] = sm.run_v[j];
        sm.cand_i[cnt + j] = sm.run_i[j];
      }
      __syncthreads();
      rank_select(sm, cnt + rn, k);
      __syncthreads();
      if (tid == 0) sm.run_n = min(k, cnt + rn);
    } else {
      // Too many ties at the threshold: exact selection by k rounds of
      // "best element strictly after the previous pick" over tile + list.
      float pv = CUDART_INF_F;
      int32_t pi = -1;
      const int rn = sm.run_n;
      int got = 0;
      for (int r = 0; r < k; ++r) {
        uint64_t best = 0;
#pragma unroll
        for (int u = 0; u < K1_U; ++u) {
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            const float xv = X(u * VEC + j);
            const int32_t xi = base + (u * K1_THREADS + tid) * VEC + j;
            if (xv > -CUDART_INF_F && better(pv, pi, xv, xi)) {
              const uint64_t key = pack_vi(xv, xi);
              best = key > best ? key : best;
            }
          }
        }
        if (tid < rn && better(pv, pi, sm.run_v[tid], sm.run_i[tid])) {
          const uint64_t key = pack_vi(sm.run_v[tid], sm.run_i[tid]);
          best = key > best ? key : best;
        }
        best = cta_max_u64(sm, best);
        if (best == 0) break;
        pv = packed_v(best);
        pi = packed_i(best);
        if (tid == 0) {
          sm.new_v[r] = pv;
          sm.new_i[r] = pi;
        }
        ++got;
      }
      __syncthreads();
      if (tid == 0) sm.run_n = got;
    }
    if (tid < k) {
      sm.run_v[tid] = sm.new_v[tid];
      sm.run_i[tid] = sm.new_i[tid];
    }
    if (tid == 0) {
      float st = 0.f;
#pragma unroll
      for (int w = 0; w < K1_WARPS; ++w) st += sm.wsum[w];
      const float mn = fmaxf(sm.run_m, mt);
      float acc = 0.f;
      if (sm.run_m > -CUDART_INF_F) acc += sm.run_s * expf(sm.run_m - mn);
      if (mt > -CUDART_INF_F) acc += st * expf(mt - mn);
      sm.run_s = acc;
      sm.run_m = mn;
      sm.cnt = 0;
    }
    __syncthreads();
  }

  // ---- cluster merge in CTA rank 0 over distributed shared memory
  cluster.sync();
  if (crank == 0) {
    __shared__ float s_thr;
    __shared__ int s_cnt;
    __shared__ float s_m;
    __shared__ float s_s;
    __shared__ float c_m[K1_MAXC], c_s[K1_MAXC], c_k[K1_MAXC];
    // one thread per cluster member reads its partial (in parallel), then
    // warp 0 reduces them
    if (tid < C) {
      const K1Smem *o = cluster.map_shared_rank(&sm, tid);
      c_m[tid] = o->run_m;
      c_s[tid] = o->run_s;
      c_k[tid] = (o->run_n == k) ? o->run_v[k - 1] : -CUDART_INF_F;
    }
    __syncthreads();
    if (tid < 32) {
      const float mc = (lane < C) ? c_m[lane] : -CUDART_INF_F;
      const float m = warp_max_f(mc);
      const float sc = warp_sum_f((lane < C && mc > -CUDART_INF_F) ? c_s[lane] * expf(mc - m) : 0.f);
      const float th = warp_max_f((lane < C) ? c_k[lane] : -CUDART_INF_F);
      if (lane == 0) {
        s_m = m;
        s_s = sc;
        s_thr = th;
        s_cnt = 0;
      }
    }
    __syncthreads();
    const float thr = s_thr;
    // gather every list entry >= thr (at least k of them exist)
    for (int e = tid; e < C * k; e += K1_THREADS) {
      const int c = e / k, j = e % k;
      const K1Smem *o = cluster.map_shared_rank(&sm, c);
      if (j < o->run_n && o->run_v[j] >= thr) {
        const int slot = atomicAdd(&s_cnt, 1);
        sm.cand_v[slot] = o->run_v[j];
        sm.cand_i[slot] = o->run_i[j];
      }
    }
    __syncthreads();
    const int M = s_cnt;
    rank_select(sm, M, k);
    __syncthreads();
    // lse = m + ln s with s = 2^e f, f in [0.5, 1): ln s = e ln 2 + ln f keeps
    // the fp32 logarithm on a small argument (absolute error ~1e-7); only the
    // final additions run in float64 (this GPU's FP64 pipe is narrow)
    int e2;
    const float f = frexpf(s_s, &e2);
    const double L = static_cast<double>(s_m) + static_cast<double>(e2) * 0.6931471805599453 +
                     static_cast<double>(logf(f));
    if (tid < k) {
      const int64_t o = static_cast<int64_t>(row) * k + tid;
      const float v = sm.new_v[tid];
      ids[o] = sm.new_i[tid];
      lg[o] = v;
      q[o] = expf(static_cast<float>(static_cast<double>(v) - L));
    }
    if (tid == 0) lse[row] = L;
  }
  cluster.sync();   // keep every CTA's shared memory alive until rank 0 is done
}

// ---------------------------------------------------------------- launcher
cudaError_t launch_topk_softmax(const void *logits, bool bf16, int rows, int V, int64_t row_stride,
                                int k, int32_t *ids, float *lg, float *q, double *lse, int num_sms,
                                cudaStream_t stream) {
  const int esz = bf16 ? 2 : 4;
  // CTAs per row: enough clusters to cover the GPU about twice, chunks of at
  // least 4096 elements, at most 16 CTAs (a non-portable cluster size).
  int C = 1;
  while (C < K1_MAXC && static_cast<int64_t>(rows) * C < 2LL * num_sms && V / (2 * C) >= 4096) C <<= 1;
  const int vec = 16 / esz;
  int chunk = (V + C - 1) / C;
  chunk = (chunk + vec - 1) / vec * vec;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((row_stride * esz) % 16 == 0);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, rows, 1);
  cfg.blockDim = dim3(K1_THREADS, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) {
    if (vec_ok)
      return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<BF16Tag, true>, logits, V, row_stride, k, chunk, ids, lg, q, lse);
    return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<BF16Tag, false>, logits, V, row_stride, k, chunk, ids, lg, q, lse);
  }
  if (vec_ok)
    return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<F32Tag, true>, logits, V, row_stride, k, chunk, ids, lg, q, lse);
  return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<F32Tag, false>, logits, V, row_stride, k, chunk, ids, lg, q, lse);
}

cudaError_t prepare_topk_softmax() {
  cudaError_t e;
  e = cudaFuncSetAttribute(topk_softmax_kernel<BF16Tag, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_softmax_kernel<BF16Tag, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_softmax_kernel<F32Tag, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topk_softmax_kernel<F32Tag, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace bst
