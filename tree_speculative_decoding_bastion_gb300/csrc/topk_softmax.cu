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
//   * one thread-block cluster of C <= 8 CTAs per drafter row; each CTA stages
//     its contiguous chunk of the row into shared memory with bulk
//     asynchronous copies (cp.async.bulk: the whole chunk in flight at once);
//   * two passes over the staged chunk: pass A finds the maxima, pass B sums
//     exp(x - max) and keeps candidates above a threshold that provably lies
//     below the chunk's k-th largest value (a per-warp sort of the lane
//     maxima); about 2k candidates survive and are ranked exactly; a chunk with
//     more than 1024 candidates (massive ties) takes k exact selection rounds;
//   * every CTA pushes its partial (max, sum, sorted top-k) into CTA rank 0's
//     shared memory with remote stores, one cluster barrier follows, and rank 0
//     merges locally and writes ids, logits, q and lse (float64 output; the
//     arithmetic is fp32 with a range-reduced logarithm).
#include <cooperative_groups.h>
#include <math_constants.h>

#include <algorithm>

#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace bst {

#ifdef BST_TRACE
__device__ unsigned long long g_k1_trace[4096 * 16];
extern "C" cudaError_t bastion_trace_read_topk(void *dst, size_t bytes) {
  return cudaMemcpyFromSymbol(dst, g_k1_trace, bytes);
}
#endif

constexpr int K1_THREADS = 512;   // 4 warps per scheduler hide the MUFU / shared-memory latency
constexpr int K1_WARPS = K1_THREADS / 32;
constexpr int K1_CAP = 1024;                      // candidate buffer
constexpr int K1_MAXC = 8;                        // CTAs per cluster (row), portable
constexpr int K1_CHUNK_BYTES = 38 * 1024;         // preferred staged bytes per CTA (8 CTAs for a 152K bf16 row)
constexpr int K1_CHUNK_BYTES_WAVES = 64 * 1024;   // when the clusters need more than one wave
constexpr int K1_CTAS_PER_SM = 4;                 // the kernel's launch bound
constexpr int K1_MAX_SMEM = 200 * 1024;           // largest chunk (very long rows)
constexpr uint64_t K1_WAIT_NS = 200ull * 1000ull * 1000ull;

struct K1Smem {
  uint64_t bar;
  float wmax[K1_WARPS];
  float wa[K1_WARPS];          // per warp: ceil(k/K1_WARPS)-th largest lane maximum
  float wb[K1_WARPS];          // per warp: k-th largest lane maximum
  float wsum[K1_WARPS];
  int cnt;
  int nres;
  float new_v[BASTION_MAX_TOPK];
  int32_t new_i[BASTION_MAX_TOPK];
  unsigned long long red[K1_WARPS];
  alignas(16) float cand_v[K1_CAP];
  alignas(16) int32_t cand_i[K1_CAP];
  // inbox of CTA rank 0: every cluster member's max, exp-sum and sorted top-k
  // (entry c * k + j; lists shorter than k are padded with (-inf, INT_MAX))
  float in_m[K1_MAXC];
  float in_s[K1_MAXC];
  alignas(16) float in_v[K1_MAXC * BASTION_MAX_TOPK];
  alignas(16) int32_t in_i[K1_MAXC * BASTION_MAX_TOPK];
  double L;
};

// Bitonic sort of one value per lane, descending (lane 0 gets the largest).
BST_DEV float warp_sort_desc(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float o = __shfl_xor_sync(FULL, v, stride);
      const bool up = ((lane & size) == 0);       // this block sorts descending
      const bool lower = ((lane & stride) == 0);  // I hold the lower index of the pair
      v = (lower == up) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

// Rank of (v, i) among the M entries (cv, ci): how many are better (value
// desc, index asc).  Four entries per 16-byte load, all loads independent.
BST_DEV int rank_among(const float *cv, const int32_t *ci, int M, float v, int32_t i) {
  int rank = 0;
  int o = 0;
#pragma unroll 4
  for (; o + 4 <= M; o += 4) {
    const float4 v4 = *reinterpret_cast<const float4 *>(cv + o);
    const int4 i4 = *reinterpret_cast<const int4 *>(ci + o);
    rank += static_cast<int>(better(v4.x, i4.x, v, i)) + static_cast<int>(better(v4.y, i4.y, v, i)) +
            static_cast<int>(better(v4.z, i4.z, v, i)) + static_cast<int>(better(v4.w, i4.w, v, i));
  }
  for (; o < M; ++o) rank += static_cast<int>(better(cv[o], ci[o], v, i));
  return rank;
}

// CTA-wide maximum of a 64-bit key (all threads get it).
BST_DEV unsigned long long cta_max_u64(K1Smem &sm, unsigned long long x) {
  x = warp_max_u64(x);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red[w] = x;
  __syncthreads();
  unsigned long long r = sm.red[0];
#pragma unroll
  for (int j = 1; j < K1_WARPS; ++j) r = sm.red[j] > r ? sm.red[j] : r;
  return r;
}

// 2^x on the special-function unit (the hardware approximation instruction)
BST_DEV float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Visit every element of the chunk owned by this thread, in increasing order:
// 16-byte vectors t, t + 256, ... from shared memory (bulk path), or scalars
// t, t + 256, ... from global memory (unaligned rows).
template <class Tag, bool kBulk, class F>
BST_DEV void for_each_elem(const uint8_t *stage, const void *rowp, int c0, int len, F &&f) {
  constexpr int VEC = Tag::kVec;
  if (kBulk) {
    const uint4 *v4 = reinterpret_cast<const uint4 *>(stage);
    const int nvec = len / VEC;
    for (int v = threadIdx.x; v < nvec; v += K1_THREADS) {
      const uint4 x = v4[v];
#pragma unroll
      for (int j = 0; j < VEC; ++j) f(elem16<Tag>(x, j), c0 + v * VEC + j);
    }
  } else {
    for (int e = threadIdx.x; e < len; e += K1_THREADS) f(load_scalar<Tag>(rowp, c0 + e), c0 + e);
  }
}

// Largest element of this thread's share of the staged chunk (16-byte
// vectors t, t + 512, ...; bf16 pairs compared packed, which is exact).
template <class Tag>
BST_DEV float staged_max(const uint8_t *stage, int len) {
  const uint4 *v4 = reinterpret_cast<const uint4 *>(stage);
  const int nvec = len / Tag::kVec;
  float m = -CUDART_INF_F;
  for (int v = threadIdx.x; v < nvec; v += K1_THREADS) m = fmaxf(m, vmax16<Tag>(v4[v]));
  return m;
}

// Pass B over the staged chunk, one 16-byte vector at a time: sum of
// exp(x - m) for this thread's elements, with x - m (exact for bf16 inputs)
// and the scale by log2(e) done on float pairs, and the candidates x >= thr
// appended to the shared list.  The per-element candidate test runs only for
// a vector whose maximum reaches thr.
template <class Tag>
BST_DEV float staged_expsum_candidates(const uint8_t *stage, int c0, int len, float m, float thr, K1Smem &sm) {
  constexpr int VEC = Tag::kVec;
  const uint4 *v4 = reinterpret_cast<const uint4 *>(stage);
  const int nvec = len / VEC;
  const float2 negm = make_float2(-m, -m);
  const float2 l2e = make_float2(kLog2e, kLog2e);
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  for (int v = threadIdx.x; v < nvec; v += K1_THREADS) {
    const uint4 x = v4[v];
    float f[VEC];
    unpack16<Tag>(x, f);
#pragma unroll
    for (int j = 0; j < VEC; j += 2) {
      const float2 t = __fmul2_rn(__fadd2_rn(make_float2(f[j], f[j + 1]), negm), l2e);
      acc[(j >> 1) & 1] = __fadd2_rn(acc[(j >> 1) & 1], make_float2(ex2f(t.x), ex2f(t.y)));
    }
    if (vmax16<Tag>(x) >= thr) {
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        if (f[j] >= thr && f[j] > -CUDART_INF_F) {
          const int slot = atomicAdd(&sm.cnt, 1);
          if (slot < K1_CAP) {
            sm.cand_v[slot] = f[j];
            sm.cand_i[slot] = c0 + v * VEC + j;
          }
        }
      }
    }
  }
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}

template <class Tag, bool kBulk>
// Four CTAs per SM (32 registers a thread): the CTAs spend most of their time
// at barriers and in their one staged copy, so more of them per SM keeps more
// bytes in flight (measured: 15.5 -> 12.9 us on 64 rows of 151936, 35.9 ->
// 33.0 us on 256 rows of 128256; a few bytes of spills).
__global__ void __launch_bounds__(K1_THREADS, K1_CTAS_PER_SM) topk_softmax_kernel(
    const void *__restrict__ logits, int V, int64_t row_stride, int k, int chunk,
    int32_t *__restrict__ ids, float *__restrict__ lg, float *__restrict__ q, double *__restrict__ lse,
    uint32_t *__restrict__ dev_err) {
  using T = typename Tag::storage;
  extern __shared__ __align__(128) uint8_t k1_stage[];
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
  const int len = max(0, min(V, c0 + chunk) - c0);
  const int kk = (k + K1_WARPS - 1) / K1_WARPS;

  if (tid == 0) BST_STAMP(g_k1_trace, 0);
  if (tid == 0) {
    sm.cnt = 0;
    if (kBulk) {
      mbar_init(&sm.bar, 1);
      fence_mbar_init();
    }
  }
  // warm L2 with this CTA's chunk while the producing grid finishes
  if (kBulk && tid == 0 && len > 0) prefetch_l2_bulk(rowp + c0, static_cast<uint32_t>(len) * sizeof(T));
  __syncthreads();
  cluster_arrive_relaxed();   // paired with the wait before the first remote store
  pdl_wait();
  pdl_trigger();
  if (tid == 0) BST_STAMP(g_k1_trace, 6);
  bool staged = true;
  if (kBulk) {
    const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
    if (tid == 0 && bytes > 0) {
      mbar_expect_tx(&sm.bar, bytes);
      for (uint32_t off = 0; off < bytes; off += 16384u)
        bulk_load(k1_stage + off, reinterpret_cast<const uint8_t *>(rowp + c0) + off, min(16384u, bytes - off), &sm.bar);
    }
    int no_abort = 0;
    if (bytes > 0 && !mbar_wait(&sm.bar, 0, &no_abort, K1_WAIT_NS)) {
      staged = false;
      if (tid == 0) set_err(dev_err, BASTION_DEVERR_TIMEOUT);
    }
  }
  const int vlen = staged ? len : 0;   // a copy that never landed counts as empty

  // ---- pass A: maxima and the candidate threshold
  float tm = -CUDART_INF_F;
  if (kBulk)
    tm = staged_max<Tag>(k1_stage, vlen);
  else
    for_each_elem<Tag, kBulk>(k1_stage, rowp, c0, vlen, [&](float x, int) { tm = fmaxf(tm, x); });
  const float sorted = warp_sort_desc(tm);
  const float a_w = __shfl_sync(FULL, sorted, kk - 1);
  const float b_w = __shfl_sync(FULL, sorted, k - 1);
  if (lane == 0) {
    sm.wmax[warp] = sorted;  // lane 0 holds the warp maximum
    sm.wa[warp] = a_w;
    sm.wb[warp] = b_w;
  }
  __syncthreads();
  if (tid == 0) BST_STAMP(g_k1_trace, 1);
  float mt = sm.wmax[0], amin = sm.wa[0], bmax = sm.wb[0];
#pragma unroll
  for (int w = 1; w < K1_WARPS; ++w) {
    mt = fmaxf(mt, sm.wmax[w]);
    amin = fminf(amin, sm.wa[w]);
    bmax = fmaxf(bmax, sm.wb[w]);
  }
  // Each warp has ceil(k/8) lane maxima >= its a_w, so >= k elements of the
  // chunk are >= min_w a_w; likewise >= k elements are >= any single b_w.
  const float thr = fmaxf(amin, bmax);

  // ---- pass B: exp-sum and candidates
  float s = 0.f;
  if (kBulk) {
    s = staged_expsum_candidates<Tag>(k1_stage, c0, vlen, mt, thr, sm);
  } else {
    for_each_elem<Tag, kBulk>(k1_stage, rowp, c0, vlen, [&](float x, int idx) {
      s += ex2f((x - mt) * kLog2e);   // exp(x - m); x - m is exact for bf16 inputs
      if (x >= thr && x > -CUDART_INF_F) {
        const int slot = atomicAdd(&sm.cnt, 1);
        if (slot < K1_CAP) {
          sm.cand_v[slot] = x;
          sm.cand_i[slot] = idx;
        }
      }
    });
  }
  s = warp_sum_f(s);
  if (lane == 0) sm.wsum[warp] = s;
  __syncthreads();
  if (tid == 0) BST_STAMP(g_k1_trace, 2);
  const int cnt = sm.cnt;
  cluster_wait();   // every CTA of the cluster has started: rank 0's shared memory exists
  K1Smem *r0 = cluster.map_shared_rank(&sm, 0);
  if (cnt <= K1_CAP) {
    // the best k candidates (ranked exactly) go straight to rank 0's inbox
    for (int c = tid; c < cnt; c += K1_THREADS) {
      const float v = sm.cand_v[c];
      const int32_t i = sm.cand_i[c];
      const int rank = rank_among(sm.cand_v, sm.cand_i, cnt, v, i);
      if (rank < k) {
        r0->in_v[crank * k + rank] = v;
        r0->in_i[crank * k + rank] = i;
      }
    }
    for (int j = cnt + tid; j < k; j += K1_THREADS) {
      r0->in_v[crank * k + j] = -CUDART_INF_F;
      r0->in_i[crank * k + j] = 0x7FFFFFFF;
    }
  } else {
    // Too many ties at the threshold: exact selection by k rounds of
    // "best element strictly after the previous pick".
    float pv = CUDART_INF_F;
    int32_t pi = -1;
    int got = 0;
    for (int r = 0; r < k; ++r) {
      unsigned long long best = 0;
      for_each_elem<Tag, kBulk>(k1_stage, rowp, c0, vlen, [&](float x, int idx) {
        if (x > -CUDART_INF_F && better(pv, pi, x, idx)) {
          const unsigned long long key = pack_vi(x, idx);
          best = key > best ? key : best;
        }
      });
      best = cta_max_u64(sm, best);
      if (best == 0) break;
      pv = packed_v(best);
      pi = packed_i(best);
      if (tid == 0) {
        // the element itself (the key maps -0.0 to +0.0)
        sm.new_v[r] = kBulk ? load_scalar_shared<Tag>(k1_stage, pi - c0) : load_scalar<Tag>(rowp, pi);
        sm.new_i[r] = pi;
      }
      ++got;
    }
    __syncthreads();
    if (tid < k) {
      r0->in_v[crank * k + tid] = tid < got ? sm.new_v[tid] : -CUDART_INF_F;
      r0->in_i[crank * k + tid] = tid < got ? sm.new_i[tid] : 0x7FFFFFFF;
    }
  }
  if (tid == 0) {
    float st = 0.f;
#pragma unroll
    for (int w = 0; w < K1_WARPS; ++w) st += sm.wsum[w];
    r0->in_m[crank] = mt;
    r0->in_s[crank] = st;
    BST_STAMP(g_k1_trace, 3);
  }
  cluster.sync();
  if (tid == 0) BST_STAMP(g_k1_trace, 4);
  if (kBulk && !staged) {
    // the staged copy timed out: let it land (bounded) before this CTA's
    // shared memory can go to another CTA
    int no_abort = 0;
    mbar_wait(&sm.bar, 0, &no_abort, K1_WAIT_NS);
  }
  if (crank != 0) return;

  // ---- rank 0: the row's lse, then the top k of the C sorted partial lists
  if (tid < 32) {
    const float mc = (lane < C) ? sm.in_m[lane] : -CUDART_INF_F;
    const float m = warp_max_f(mc);
    const float sc = warp_sum_f((lane < C && mc > -CUDART_INF_F) ? sm.in_s[lane] * expf(mc - m) : 0.f);
    if (lane == 0) {
      // lse = m + ln s with s = 2^e f, f in [0.5, 1): ln s = e ln 2 + ln f keeps
      // the fp32 logarithm on a small argument (absolute error ~1e-7); only the
      // final additions run in float64 (this GPU's FP64 pipe is narrow)
      int e2;
      const float f = frexpf(sc, &e2);
      sm.L = static_cast<double>(m) + static_cast<double>(e2) * 0.6931471805599453 + static_cast<double>(logf(f));
    }
  }
  __syncthreads();
  const double L = sm.L;
  const int M = C * k;
  for (int e = tid; e < M; e += K1_THREADS) {
    const float v = sm.in_v[e];
    const int32_t i = sm.in_i[e];
    if (v == -CUDART_INF_F) continue;
    const int rank = rank_among(sm.in_v, sm.in_i, M, v, i);
    if (rank < k) {
      const int64_t o = static_cast<int64_t>(row) * k + rank;
      ids[o] = i;
      lg[o] = v;
      q[o] = expf(static_cast<float>(static_cast<double>(v) - L));
    }
  }
  if (tid == 0) {
    lse[row] = L;
    BST_STAMP(g_k1_trace, 5);
  }
}

// ---------------------------------------------------------------- launcher
cudaError_t launch_topk_softmax(const void *logits, bool bf16, int rows, int V, int64_t row_stride, int k,
                                int32_t *ids, float *lg, float *q, double *lse, uint32_t *dev_err, int num_sms,
                                cudaStream_t stream) {
  const int esz = bf16 ? 2 : 4;
  const int vec = 16 / esz;
  // CTAs per row: staged chunks of about 38 KB, at most a portable cluster of 8
  // (very long rows take larger chunks).  When the rows' clusters do not fit
  // in one wave of resident CTAs, chunks of up to 64 KB (three CTAs per SM):
  // fewer, longer CTAs take fewer waves (measured: 256 rows of 128256,
  // 35.4 -> 31.7 us with 64 KB, 33.3 with 48 KB; 128 rows of 151936,
  // 24.9 -> 23.2 us), while a single wave is faster with the smaller chunks
  // (64 rows of 151936: 14.0 us against 14.5 with 48 KB).
  const int64_t row_bytes = static_cast<int64_t>(V) * esz;
  auto ctas_per_row = [&](int64_t chunk_bytes) {
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(K1_MAXC, (row_bytes + chunk_bytes - 1) / chunk_bytes)));
  };
  int C = ctas_per_row(K1_CHUNK_BYTES);
  if (num_sms > 0 && static_cast<int64_t>(rows) * C > static_cast<int64_t>(K1_CTAS_PER_SM) * num_sms)
    C = ctas_per_row(K1_CHUNK_BYTES_WAVES);
  int chunk = (V + C - 1) / C;
  chunk = (chunk + vec - 1) / vec * vec;
  C = (V + chunk - 1) / chunk;
  const bool bulk = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((row_stride * esz) % 16 == 0) &&
                    (row_bytes % 16 == 0) && (static_cast<int64_t>(chunk) * esz <= K1_MAX_SMEM);

  const size_t dyn = bulk ? static_cast<size_t>(chunk) * esz : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, rows, 1);
  cfg.blockDim = dim3(K1_THREADS, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = fill_launch_attrs(attr, C, 1);
#define BST_K1_ARGS logits, V, row_stride, k, chunk, ids, lg, q, lse, dev_err
  if (bf16) {
    if (bulk) return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<BF16Tag, true>, BST_K1_ARGS);
    return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<BF16Tag, false>, BST_K1_ARGS);
  }
  if (bulk) return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<F32Tag, true>, BST_K1_ARGS);
  return cudaLaunchKernelEx(&cfg, topk_softmax_kernel<F32Tag, false>, BST_K1_ARGS);
#undef BST_K1_ARGS
}

cudaError_t prepare_topk_softmax() {
  cudaError_t e;
  const void *fns[2][2] = {{reinterpret_cast<const void *>(topk_softmax_kernel<F32Tag, false>),
                            reinterpret_cast<const void *>(topk_softmax_kernel<F32Tag, true>)},
                           {reinterpret_cast<const void *>(topk_softmax_kernel<BF16Tag, false>),
                            reinterpret_cast<const void *>(topk_softmax_kernel<BF16Tag, true>)}};
  for (int b = 0; b < 2; ++b)
    for (int u = 0; u < 2; ++u) {
      e = cudaFuncSetAttribute(fns[b][u], cudaFuncAttributeMaxDynamicSharedMemorySize, K1_MAX_SMEM);
      if (e != cudaSuccess) return e;
      if ((e = prefer_max_shared(fns[b][u])) != cudaSuccess) return e;
    }
  return cudaSuccess;
}

}  // namespace bst
