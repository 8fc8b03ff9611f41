// Stage 3: tree-masked verification attention of the tree tokens.
//
// "Bastion: Budget-Aware Speculative Decoding with Tree-structured Block
// Diffusion Drafting" (explainer gist.science/de/paper/2605.29727),
// "Problemstellung": the target model verifies the drafted candidates in one
// parallel pass; "Akzeptanzlänge": the verification is tree-structured.  For
// every tree node i and query head h the target attends to the whole context
// and to the tree tokens on the root-to-i path (the ancestor bitmask of
// stage 2, self included):
//     out = softmax(q . keys * scale) . values.
//
// bf16 path (tcgen05, S / P / O in tensor memory): the 128 M rows of a unit
// pack g = Hq/Hkv query heads x tree nodes of one KV head (GQA), so every K/V
// tile of 128 keys is used by all heads of its group.  Two kernels:
//   * contiguous caches: one CTA per (request, KV head, M-tile, KV split),
//     the splits of a unit forming a cluster that merges through L2;
//   * paged caches: one CTA per SM streaming an equal share of the batch's
//     concatenated tiles in gangs, units cut between gangs merged by the CTA
//     that takes a unit's last ticket.
// Details at each kernel.
//
// f32 path: an exact fp32 flash-decoding kernel, one CTA per (b, node, head),
// 128-key blocks staged in shared memory.
#include <math_constants.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "sm100_ptx.cuh"

namespace bst {

constexpr int ATT_THREADS = 320;        // 8 softmax warps, a TMA warp, an MMA warp
constexpr int ATT_SM_THREADS = 256;     // softmax threads
constexpr int ATT_TMA_WARP = 8;
constexpr int ATT_MMA_WARP = 9;
constexpr int ATT_N = 128;              // keys per tile
constexpr int ATT_M = 128;              // rows per M-tile
constexpr int ATT_HALF = ATT_N * 128;   // bytes of 128 rows x 64 bf16
constexpr int ATT_SBUF = 3;             // S / P buffers in TMEM (128 columns each; O follows)
constexpr int ATT_MAX_STAGES = 3;
constexpr int ATT_MAX_B = 512;          // requests per call (their cost prefix lives in shared memory)
constexpr int ATT_MIN_SHARE = 8;        // tiles of a gang's range at least (unless the batch has fewer)
constexpr uint64_t ATT_WAIT_NS = 200ull * 1000ull * 1000ull;
constexpr float ATT_RESCALE_LOG2 = 8.f;

struct PagedParams {
  int B, n_max, Hq, Hkv, g, mt_max;   // mt_max: 128-row M-tiles of a (request, KV head) at n_max
  int nctas;                          // CTAs of the grid (the work is split evenly over them)
  float scale_log2;                   // scale * log2(e)
  int page_size, max_pages, num_pages;
  int64_t cap;                        // context capacity per request
  const int32_t *ctx_len;
  const int32_t *n;
  const unsigned long long *mask;
  const int32_t *block_table;
  uint16_t *out;                      // bf16 [B, n_max, Hq, d]
  uint32_t *tickets;                  // [B * Hkv * mt_max], zero between calls
  float4 *part;                       // [nctas][2] partial (O, m, l) slots
  uint32_t *dev_err;
};

struct PagedBars {
  uint64_t q_full;
  uint64_t q_free;                    // the last S of a unit finished: Q may be replaced
  uint64_t o_free;                    // the softmax read O of a unit: the next unit's P V may start
  uint64_t o_full;                    // a unit's last P V finished: O is final (one phase per unit)
  uint64_t k_full[ATT_MAX_STAGES];
  uint64_t k_empty[ATT_MAX_STAGES];   // S(j) finished: K stage j mod KS free
  uint64_t v_full[ATT_MAX_STAGES];
  uint64_t v_empty[ATT_MAX_STAGES];   // P V(j) finished (V stage j free, O updated)
  uint64_t s_full[ATT_SBUF];          // S(j) finished (S ready for the softmax)
  uint64_t p_full[ATT_SBUF];
  uint64_t drain;
  uint64_t part_done;                 // every softmax thread stored its share of a partial
  uint64_t part_go;                   // the ticket of that partial was taken
  // the two softmax warps that share a row quarter (warps q and q + 4, one
  // half of the columns each) swap their row maxima every tile, and their
  // row sums at the end of a unit, through xmax / xl; xbar[q] completes once
  // per swap
  uint64_t xbar[4];
  float xmax[2][2][ATT_M];            // [swap parity][column half][row]
  float xl[2][ATT_M];                 // [column half][row]
  int last_piece;                     // this CTA completes the unit whose partial it just stored
  int gang_g, gang_n, my_tiles;       // gang size, gangs, tiles of this CTA
  uint32_t tmem_base;
  int abort;
  int64_t pre[ATT_MAX_B + 1];         // prefix over requests of (units x tiles)
};

template <int D>
struct PagedLayout {
  static constexpr int NH = D / 64;
  // A V tile is needed only after the softmax's P, three tiles after its K
  // (S runs ahead), so V gets the deeper ring: with head_dim 128 three V
  // tiles and two K tiles fit next to Q and the barriers.  (Measured on the
  // 4 x 32K-context batch: a V tile lands about 1.6 us after its copy
  // starts, and with two V stages the copy of V(j) waits for P V(j - 2), so
  // a tile took about 1 us.)
  static constexpr int KSTAGES = D == 128 ? 2 : 3;
  static constexpr int VSTAGES = 3;
  static constexpr int Q_BYTES = NH * ATT_HALF;
  static constexpr int KV_BYTES = NH * ATT_HALF;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_BYTES;
  static constexpr int V_OFF = K_OFF + KSTAGES * KV_BYTES;
  static constexpr int BAR_OFF = V_OFF + VSTAGES * KV_BYTES;

  static constexpr int USED = BAR_OFF + static_cast<int>(sizeof(PagedBars));
  // 1024 bytes of slack for aligning the dynamic shared memory base; at least
  // 120 KB so that a single CTA owns each SM (its TMEM allocation is 512 columns).
  static constexpr int SMEM = (USED + 1024) > 120 * 1024 ? (USED + 1024) : 120 * 1024;
  static_assert(SMEM <= 227 * 1024, "exceeds the shared memory of one CTA");
  static_assert(ATT_SBUF * 128 + D <= 512, "S buffers and O must fit the 512 TMEM columns");
};

// Optional phase trace (compiled in with -DBST_TRACE only): %globaltimer
// stamps at the pipeline's phase boundaries, 64 per CTA, read back with
// bastion_trace_read().  Normal builds contain none of it.
#ifdef BST_TRACE
__device__ unsigned long long g_attn_trace[4096 * 64];
#define BST_TRACE_AT(ev)                                                                                  \
  do {                                                                                                  \
    const unsigned cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);               \
    if (cta_ < 4096u && (ev) < 64) g_attn_trace[cta_ * 64u + (ev)] = globaltimer_ns();                 \
  } while (0)
extern "C" cudaError_t bastion_trace_read(void *dst, size_t bytes) {
  return cudaMemcpyFromSymbol(dst, g_attn_trace, bytes);
}
#else
#define BST_TRACE_AT(ev) \
  do {                   \
  } while (0)
#endif

// all threads of the warp agree on the outcome of a bounded wait
BST_DEV bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = mbar_wait(bar, parity, abort, ATT_WAIT_NS);
  return __all_sync(FULL, ok);
}

BST_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^x on the special-function unit (the hardware approximation instruction;
// 2^-inf = 0)
BST_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- softmax steps
// (shared by both kernels: one softmax warp, one 128-key tile, this warp's
// row quarter and column half)

// This warp's 64 S columns of the tile, masked (a context tile: keys from
// nvalid on are past the context; a tree tile: bit c of wb marks an ancestor
// or the node itself), and their maximum.
BST_DEV float softmax_load_mask_max(uint32_t taddr, bool is_ctx, int nvalid, unsigned long long wb,
                                    uint32_t (&s)[ATT_N / 2]) {
  constexpr int HC = ATT_N / 2;
  tmem_ld32(taddr + 0, s + 0);
  tmem_ld32(taddr + 32, s + 32);
  tmem_wait_ld32(s + 0);
  tmem_wait_ld32(s + 32);
  // masked scores become -inf
  const uint32_t NEG = 0xff800000u;
  if (is_ctx) {
    if (nvalid < HC) {
#pragma unroll
      for (int c = 0; c < HC; ++c) s[c] = (c < nvalid) ? s[c] : NEG;
    }
  } else {
#pragma unroll
    for (int c = 0; c < HC; ++c) s[c] = ((wb >> c) & 1ull) ? s[c] : NEG;
  }
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
  for (int c = 8; c < HC; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(s[c]));
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// P = 2^(S cs - msub) as bf16 pairs into TMEM at taddr_p (32 columns), and
// the sum of this half-row's P (before rounding).  The softmax warps are
// bound by instruction issue, so the scale-and-offset and the sums run on
// packed fp32 pairs (FFMA2, FADD2): long_ctx_b4 attention 271 -> 253 us.
BST_DEV float softmax_exp_store(const uint32_t (&s)[ATT_N / 2], float cs, float msub, uint32_t taddr_p) {
  constexpr int HC = ATT_N / 2;
  float2 sum[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sum[i] = make_float2(0.f, 0.f);
  uint32_t pk[HC / 2];
  const float2 cs2 = make_float2(cs, cs), ms2 = make_float2(-msub, -msub);
#pragma unroll
  for (int c = 0; c < HC; c += 2) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), cs2, ms2);
    const float p0 = ex2(x.x);
    const float p1 = ex2(x.y);
    sum[(c >> 1) & 3] = __fadd2_rn(sum[(c >> 1) & 3], make_float2(p0, p1));
    pk[c >> 1] = pack_bf16x2(p0, p1);
  }
  tmem_st32(taddr_p, pk);
  return ((sum[0].x + sum[1].x) + (sum[2].x + sum[3].x)) + ((sum[0].y + sum[1].y) + (sum[2].y + sum[3].y));
}

// O *= alpha on this warp's DH columns of its rows.
template <int DH>
BST_DEV void rescale_o(uint32_t taddr, float alpha) {
#pragma unroll
  for (int cc = 0; cc < DH / 32; ++cc) {
    uint32_t o[32];
    tmem_ld32(taddr + cc * 32, o);
    tmem_wait_ld32(o);
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
    tmem_st32(taddr + cc * 32, o);
  }
}

// This warp's DH columns of O for its row.
template <int DH>
BST_DEV void load_o(uint32_t taddr, float *o) {
#pragma unroll
  for (int cc = 0; cc < DH / 32; ++cc) {
    uint32_t t32[32];
    tmem_ld32(taddr + cc * 32, t32);
    tmem_wait_ld32(t32);
#pragma unroll
    for (int e = 0; e < 32; ++e) o[cc * 32 + e] = __uint_as_float(t32[e]);
  }
}

// One softmax thread's output: GQA row `row` of (request b, KV head kvh),
// columns [D/2 ch, D/2 ch + D/2), scaled by inv.
template <int D>
BST_DEV void store_out_half(uint16_t *out, int n_max, int Hq, int g, int b, int kvh, int row, int ch, const float *o,
                            float inv) {
  constexpr int DH = D / 2;
  const int node = row / g;
  const int hl = row - node * g;
  uint16_t *dst = out + ((static_cast<int64_t>(b) * n_max + node) * Hq + kvh * g + hl) * D + ch * DH;
#pragma unroll
  for (int c = 0; c < DH; c += 8) {
    uint4 v;
    v.x = pack_bf16x2(o[c + 0] * inv, o[c + 1] * inv);
    v.y = pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
    v.z = pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
    v.w = pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
    *reinterpret_cast<uint4 *>(dst + c) = v;
  }
}

// ================================================================ contiguous
// caches: one CTA per (request, KV head, 128-row M-tile, KV split)
//
// A request's context tiles followed by its tree tiles are spread evenly over
// S KV splits; the S CTAs of one (request, KV head, M-tile) form a cluster:
// each stores its partial (O, m, l) to the workspace in L2, one cluster
// barrier publishes them, and every CTA merges a slice of the rows.  The M
// tiles of a (request, KV head) read the same K/V tiles at about the same
// time, so each tile crosses from HBM into L2 once.  Roles as in the paged
// kernel below (warp 8 TMA, warp 9 MMA, warps 0-7 softmax), one unit per CTA.
constexpr int ATT_MAX_SPLITS = 16;      // cluster size; above 8 (non-portable) where the device keeps them resident

struct SplitParams {
  int B, n_max, Hq, Hkv, g, mtiles, splits;
  float scale_log2;          // scale * log2(e)
  int64_t cap;               // context capacity per request
  const int32_t *ctx_len;
  const int32_t *n;
  const unsigned long long *mask;
  uint16_t *out;             // bf16 [B, n_max, Hq, d]
  float4 *part;              // split partials (workspace), used when splits > 1
  uint32_t *dev_err;
};

struct SplitBars {
  uint64_t q_full;
  uint64_t k_full[ATT_SBUF];
  uint64_t v_full[ATT_MAX_STAGES];
  uint64_t v_empty[ATT_MAX_STAGES];   // P V(j) finished (V stage j free, O updated)
  uint64_t s_full[ATT_SBUF];          // S(j) finished (S ready, K stage j mod 3 free)
  uint64_t p_full[ATT_SBUF];
  uint64_t drain;
  uint64_t xbar[4];                   // half-row max / sum swaps of warps q and q + 4
  float xmax[2][2][ATT_M];
  // (the row sums' swap at the end, [column half][row], uses the first K
  // stage: by then every MMA has read its last K tile)
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct SplitLayout {
  static constexpr int NH = D / 64;
  static constexpr int KSTAGES = ATT_SBUF;   // K stage j mod 3 is S buffer j mod 3 (one barrier serves both)
  // Three V stages too: with two, the copy of V(j) could start only once
  // P V(j - 2) had freed its stage, so a tile took at least half a load
  // latency.  With head_dim 128 the seven 32 KB tiles leave 3 KB of the
  // 227 KB for the barriers, so the dynamic shared memory is used unpadded
  // (its base is 1024-byte aligned: the kernel has no static shared memory)
  // and the row sums swap through a K stage at the end.
  static constexpr int VSTAGES = 3;
  static constexpr int KV_BYTES = NH * ATT_HALF;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = NH * ATT_HALF;
  static constexpr int V_OFF = K_OFF + KSTAGES * KV_BYTES;
  static constexpr int BAR_OFF = V_OFF + VSTAGES * KV_BYTES;
  static constexpr int USED = BAR_OFF + static_cast<int>(sizeof(SplitBars));
  // at least 120 KB so that a single CTA owns each SM (its TMEM allocation is 512 columns)
  static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
  static_assert(SMEM <= 227 * 1024, "exceeds the shared memory of one CTA");
};

// KV-split partials live in the workspace, one slot per (b, kvh, M-tile,
// split): (D/4 + 1) x 128 float4, column-major by float4; the last chunk of a
// row holds (m, l, 0, 0) with m in the log2 domain.
template <int D>
BST_DEV float4 *split_slot(const SplitParams &p, int b, int kvh, int mtile, int split) {
  const int64_t slot = ((static_cast<int64_t>(b) * p.Hkv + kvh) * p.mtiles + mtile) * p.splits + split;
  return p.part + slot * (D / 4 + 1) * ATT_M;
}

// Merge of the S split partials (every CTA of the cluster, after a cluster
// barrier that follows all main loops and partial stores).  CTA `split` owns
// R = ceil(128 / S) rows of the M-tile: O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s.  G threads share a row, each taking CPG of its D/4
// float4 columns; every load is issued before any is used (one L2 round trip).
template <int D, int S>
BST_DEV void merge_splits(const SplitParams &p, int b, int kvh, int mtile, int split, int nb) {
  constexpr int R = (ATT_M + S - 1) / S;
  constexpr int G = ATT_THREADS / R;
  constexpr int NC4 = D / 4;
  constexpr int CPG = (NC4 + G - 1) / G;
  const int tid = threadIdx.x;
  if (tid >= R * G) return;
  const int rl = tid % R;
  const int rr = split * R + rl;
  if (rr >= ATT_M) return;
  const int gi = tid / R;
  const int c40 = gi * CPG;
  const int prow = mtile * ATT_M + rr;
  const int nd = prow / p.g;
  if (nd >= nb) return;
  float4 ml[S];
  float4 ov[S][CPG];
#pragma unroll
  for (int s2 = 0; s2 < S; ++s2) {
    const float4 *src = split_slot<D>(p, b, kvh, mtile, s2);
    ml[s2] = __ldcg(src + NC4 * ATT_M + rr);
#pragma unroll
    for (int c = 0; c < CPG; ++c)
      ov[s2][c] = (c40 + c < NC4) ? __ldcg(src + (c40 + c) * ATT_M + rr) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = -CUDART_INF_F;
#pragma unroll
  for (int s2 = 0; s2 < S; ++s2) M = fmaxf(M, ml[s2].x);
  float4 acc[CPG];
#pragma unroll
  for (int c = 0; c < CPG; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
#pragma unroll
  for (int s2 = 0; s2 < S; ++s2) {
    // empty splits carry m = -inf, l = 0 and a zero O
    const float w = (ml[s2].x == -CUDART_INF_F) ? 0.f : ex2(ml[s2].x - M);
    lsum += w * ml[s2].y;
#pragma unroll
    for (int c = 0; c < CPG; ++c) {
      acc[c].x += w * ov[s2][c].x;
      acc[c].y += w * ov[s2][c].y;
      acc[c].z += w * ov[s2][c].z;
      acc[c].w += w * ov[s2][c].w;
    }
  }
  const float inv = 1.f / lsum;
  const int hl = prow - nd * p.g;
  uint16_t *dst = p.out + ((static_cast<int64_t>(b) * p.n_max + nd) * p.Hq + kvh * p.g + hl) * D;
#pragma unroll
  for (int c = 0; c < CPG; ++c) {
    if (c40 + c < NC4) {
      uint2 v;
      v.x = pack_bf16x2(acc[c].x * inv, acc[c].y * inv);
      v.y = pack_bf16x2(acc[c].z * inv, acc[c].w * inv);
      *reinterpret_cast<uint2 *>(dst + (c40 + c) * 4) = v;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1) tree_attn_split_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kt,
    const __grid_constant__ CUtensorMap tm_vt, const SplitParams p) {
  using LY = SplitLayout<D>;
  constexpr int KS = LY::KSTAGES;
  constexpr int VS = LY::VSTAGES;
  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzled TMA tiles need a 1024-byte aligned base, which the
  // unpadded layout takes as given; a misaligned base is reported, not used
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) set_err(p.dev_err, BASTION_DEVERR_LAYOUT);
    return;
  }
  uint8_t *smem = smem_raw;
  uint8_t *sQ = smem + LY::Q_OFF;
  SplitBars *bars = reinterpret_cast<SplitBars *>(smem + LY::BAR_OFF);
  float *xl = reinterpret_cast<float *>(smem + LY::K_OFF);   // [2][ATT_M], used after the last MMA
  volatile int *abort = &bars->abort;

  const int mtile = blockIdx.x;
  const int split = blockIdx.y;   // the cluster spans the splits (blockIdx.y)
  const int bh = blockIdx.z;
  const int b = bh / p.Hkv;
  const int kvh = bh - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  if (tid == 0) BST_TRACE_AT(0);
  // private set-up first (barriers, descriptor prefetch), then the wait for
  // the grid that produced the tree
  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
#pragma unroll
    for (int i = 0; i < KS; ++i) mbar_init(&bars->k_full[i], 1);
#pragma unroll
    for (int i = 0; i < VS; ++i) mbar_init(&bars->v_full[i], 1), mbar_init(&bars->v_empty[i], 1);
#pragma unroll
    for (int i = 0; i < ATT_SBUF; ++i) mbar_init(&bars->s_full[i], 1), mbar_init(&bars->p_full[i], ATT_SM_THREADS);
    mbar_init(&bars->drain, 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(&bars->xbar[i], 64);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == ATT_TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_kt);
    tma_prefetch_desc(&tm_vt);
  }
  pdl_wait();
  pdl_trigger();
  // request-level checks: identical for every CTA of a cluster, so a cluster
  // leaves together
  const int nb = p.n[b];
  if (nb < 1 || nb > p.n_max) {
    if (tid == 0 && mtile == 0 && split == 0 && kvh == 0) set_err(p.dev_err, BASTION_DEVERR_N);
    return;
  }
  int L = p.ctx_len[b];
  if (L < 0 || L > p.cap) {
    if (tid == 0 && mtile == 0 && split == 0 && kvh == 0) set_err(p.dev_err, BASTION_DEVERR_CTX);
    L = L < 0 ? 0 : static_cast<int>(p.cap);
  }
  if (mtile * ATT_M >= nb * p.g) return;   // no active row in this M-tile

  // the request's context tiles followed by its tree tiles, spread evenly
  // over the splits: this split takes tiles [g0, g1)
  const int ctx_tiles = (L + ATT_N - 1) / ATT_N;
  const int tot_tiles = ctx_tiles + (nb + ATT_N - 1) / ATT_N;
  const int g0 = (split * tot_tiles) / p.splits;
  const int g1 = ((split + 1) * tot_tiles) / p.splits;
  const int ct0 = g0;                                     // first context tile
  const int n_ctx = max(0, min(g1, ctx_tiles) - g0);
  const int tr0 = max(g0, ctx_tiles) - ctx_tiles;         // first tree tile
  const int n_tree = max(0, g1 - max(g0, ctx_tiles));
  const int T = n_ctx + n_tree;

  // row owned by a softmax thread (warps 0-7: row tid mod 128, column half
  // tid / 128)
  const int r = tid & (ATT_M - 1);
  const int pidx = mtile * ATT_M + r;
  const int node = pidx / p.g;
  const bool active = (tid < 2 * ATT_M) && (node < nb);

  float m_run = -CUDART_INF_F;
  float l_run = 0.f;
  bool ok = true;
  uint32_t tbase = 0;

  if (T > 0 && warp == 0) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) BST_TRACE_AT(1);

  if (T > 0) {
    tbase = bars->tmem_base;
    const uint32_t tO = tbase + ATT_SBUF * 128;

    if (warp == ATT_TMA_WARP) {
      // ------------------------------------------------ TMA producer
      if (lane == 0) {
        BST_TRACE_AT(2);
        mbar_expect_tx(&bars->q_full, LY::NH * ATT_HALF);
#pragma unroll
        for (int h = 0; h < LY::NH; ++h)
          tma_load_3d(sQ + h * ATT_HALF, &tm_q, &bars->q_full, h * 64, kvh * p.g, b * p.n_max + mtile * (ATT_M / p.g));
        // one K or V tile (context or tree) into `dst`, completing on `fb`
        auto load_tile = [&](int j, bool is_v, uint8_t *dst, uint64_t *fb) {
          if (j < n_ctx) {
#pragma unroll
            for (int h = 0; h < LY::NH; ++h)
              tma_load_3d(dst + h * ATT_HALF, is_v ? &tm_v : &tm_k, fb, h * 64, (ct0 + j) * ATT_N, b * p.Hkv + kvh);
          } else {
            const int tt = tr0 + j - n_ctx;
#pragma unroll
            for (int h = 0; h < LY::NH; ++h)
              tma_load_3d(dst + h * ATT_HALF, is_v ? &tm_vt : &tm_kt, fb, h * 64, kvh, b * p.n_max + tt * ATT_N);
          }
        };
        int k_issued = 0, v_issued = 0;
        auto issue_k = [&](int j) -> bool {
          const int st = j % KS;
          // the stage is free once S(j - KS), which read it, is complete
          if (j >= KS && !mbar_wait(&bars->s_full[st], ((j / KS) - 1) & 1, abort, ATT_WAIT_NS)) return false;
          mbar_expect_tx(&bars->k_full[st], LY::KV_BYTES);
          load_tile(j, false, smem + LY::K_OFF + st * LY::KV_BYTES, &bars->k_full[st]);
          if (j < 8) BST_TRACE_AT(32 + j);
          k_issued = j + 1;
          return true;
        };
        auto issue_v = [&](int j) -> bool {
          const int st = j % VS;
          if (j >= VS && !mbar_wait(&bars->v_empty[st], ((j / VS) - 1) & 1, abort, ATT_WAIT_NS)) return false;
          mbar_expect_tx(&bars->v_full[st], LY::KV_BYTES);
          load_tile(j, true, smem + LY::V_OFF + st * LY::KV_BYTES, &bars->v_full[st]);
          if (j < 8) BST_TRACE_AT(48 + j);
          v_issued = j + 1;
          return true;
        };
        // K runs one tile ahead of V
        bool run = issue_k(0);
        for (int j = 0; run && j < T; ++j) {
          if (j + 1 < T && !issue_k(j + 1)) break;
          if (!issue_v(j)) break;
        }
        if (*abort) {
          // let the copies already in flight land before the CTA goes away
          for (int j = max(0, k_issued - KS); j < k_issued; ++j)
            mbar_wait(&bars->k_full[j % KS], (j / KS) & 1, abort, ATT_WAIT_NS);
          for (int j = max(0, v_issued - VS); j < v_issued; ++j)
            mbar_wait(&bars->v_full[j % VS], (j / VS) & 1, abort, ATT_WAIT_NS);
          mbar_wait(&bars->q_full, 0, abort, ATT_WAIT_NS);
        }
      }
    } else if (warp == ATT_MMA_WARP) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t IDESC_QK = idesc_bf16(ATT_M, ATT_N, 0);
        constexpr uint32_t IDESC_PV = idesc_bf16(ATT_M, D, 1);
        // descriptors at the bases of Q, K stage 0 and V stage 0; a
        // descriptor's start address is its low 14 bits (address >> 4)
        const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t kdesc0 = sdesc_sw128(smem_u32(smem + LY::K_OFF), 16, 1024);
        const uint64_t vdesc0 = sdesc_sw128(smem_u32(smem + LY::V_OFF), ATT_HALF, 1024);
        bool any = false;
        // S(jj) into S buffer jj mod 3, which is also K stage jj mod 3: one
        // commit tells the softmax that S is ready and the producer that the K
        // stage is free
        auto issue_qk = [&](int jj) -> bool {
          const int ks = jj % KS;
          if (!mbar_wait(&bars->k_full[ks], (jj / KS) & 1, abort, ATT_WAIT_NS)) return false;
          if (jj < 8) BST_TRACE_AT(40 + jj);
          tc_fence_after();
          const uint64_t kdesc = kdesc0 + static_cast<uint64_t>((ks * LY::KV_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * ATT_HALF + (kk & 3) * 32) >> 4);
            mma_ss(tbase + ks * 128, qdesc0 + off, kdesc + off, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          any = true;
          mma_commit(&bars->s_full[ks]);
          BST_TRACE_AT(3 + min(jj, 7));
          return true;
        };
        // O += P(jj) V(jj); one commit frees the V stage and tells the softmax
        // that O holds P(jj) V(jj)
        auto issue_pv = [&](int jj) -> bool {
          const int sb = jj % ATT_SBUF;
          const int vs = jj % VS;
          if (!mbar_wait(&bars->p_full[sb], (jj / ATT_SBUF) & 1, abort, ATT_WAIT_NS)) return false;
          if (!mbar_wait(&bars->v_full[vs], (jj / VS) & 1, abort, ATT_WAIT_NS)) return false;
          if (jj < 8) BST_TRACE_AT(56 + jj);
          tc_fence_after();
          // V is the MN-major B operand: 8 keys per 1024-byte swizzle group,
          // the two 64-column halves of d ATT_HALF bytes apart
          const uint64_t vdesc = vdesc0 + static_cast<uint64_t>((vs * LY::KV_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < ATT_N / 16; ++kk)
            mma_ts(tO, tbase + sb * 128 + kk * 8, vdesc + static_cast<uint64_t>((kk * 2048) >> 4), IDESC_PV,
                   (jj > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->v_empty[vs]);
          return true;
        };
        bool run = mbar_wait(&bars->q_full, 0, abort, ATT_WAIT_NS);
        tc_fence_after();
        // S runs three tiles ahead of P V: S(j + 3) reuses the buffer of
        // S(j) / P(j) and is issued after P V(j), which read P(j) there (the
        // tcgen05.mma of one thread execute in issue order)
        for (int j = 0; run && j < min(T, ATT_SBUF); ++j) run = issue_qk(j);
        for (int j = 0; run && j < T; ++j) {
          if (!issue_pv(j)) { run = false; break; }
          if (j + ATT_SBUF < T && !issue_qk(j + ATT_SBUF)) { run = false; break; }
        }
        if (any) {
          // every MMA issued above has finished before TMEM is released
          mma_commit(&bars->drain);
          mbar_wait(&bars->drain, 0, abort, ATT_WAIT_NS);
        }
      }
    } else {
      // ------------------------------------------------ softmax warps 0-7
      constexpr int HC = ATT_N / 2;    // S columns per warp
      constexpr int DH = D / 2;        // O columns per warp
      const int rq = warp & 3;
      const int ch = warp >> 2;
      const uint32_t lane_off = static_cast<uint32_t>(rq * 32) << 16;
      const int W = (p.n_max + 63) >> 6;
      unsigned long long mw[4] = {0ull, 0ull, 0ull, 0ull};
      if (active) {
        const unsigned long long *mrow = p.mask + (static_cast<int64_t>(b) * p.n_max + node) * W;
        for (int w = 0; w < W; ++w) mw[w] = mrow[w];
      }
      const float cs = p.scale_log2;
      uint64_t *xb = &bars->xbar[rq];
      for (int j = 0; j < T; ++j) {
        const int sb = j % ATT_SBUF;
        if (!warp_wait(&bars->s_full[sb], (j / ATT_SBUF) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        if (tid == 0) BST_TRACE_AT(11 + min(j, 7));
        uint32_t s[HC];
        const bool is_ctx = j < n_ctx;
        const int nvalid = is_ctx ? L - (ct0 + j) * ATT_N - ch * HC : 0;
        const unsigned long long wb = is_ctx ? 0ull : mw[2 * (tr0 + j - n_ctx) + ch];
        float hmax = softmax_load_mask_max(tbase + lane_off + sb * 128 + ch * HC, is_ctx, nvalid, wb, s);
        // swap half maxima with the partner warp; the arrival also tells it
        // this warp's TMEM loads of S are complete (its P stores may then
        // overwrite those columns)
        bars->xmax[j & 1][ch][r] = hmax;
        tc_fence_before();
        mbar_arrive(xb);
        if (!warp_wait(xb, j & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const float tmax = fmaxf(hmax, bars->xmax[j & 1][ch ^ 1][r]) * cs;
        const float m_new = fmaxf(m_run, tmax);
        // keep the running reference unless the max grew by more than 2^8
        const bool jump = m_new > m_run + ATT_RESCALE_LOG2;
        const float m_use = jump ? m_new : m_run;
        const float alpha = jump ? ex2(m_run - m_new) : 1.f;
        l_run = l_run * alpha + softmax_exp_store(s, cs, (m_use == -CUDART_INF_F) ? 0.f : m_use,
                                                  tbase + lane_off + sb * 128 + ch * (HC / 2));
        const bool need = (j >= 1) && jump && (m_run > -CUDART_INF_F);
        if (__any_sync(FULL, need)) {
          // O must hold P_{j-1} V_{j-1} before it is rescaled (that P V's commit
          // arrives on its V stage's barrier, which is at most one phase
          // behind: S(j) is complete, so P V(j - 3) and every earlier MMA are too)
          if (!warp_wait(&bars->v_empty[(j - 1) % VS], ((j - 1) / VS) & 1, abort)) { ok = false; break; }
          tc_fence_after();
          rescale_o<DH>(tO + lane_off + ch * DH, alpha);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
        if (tid == 0) BST_TRACE_AT(19 + min(j, 7));
        m_run = m_use;
      }
      // ---- epilogue: O after the last P V (the drain barrier completes once,
      // after every MMA of this CTA); the two halves' row sums add
      if (ok && !warp_wait(&bars->drain, 0, abort)) ok = false;
      if (tid == 0) BST_TRACE_AT(27);
      xl[ch * ATT_M + r] = l_run;
      mbar_arrive(xb);
      if (ok && !warp_wait(xb, T & 1, abort)) ok = false;
      const float l_row = l_run + xl[(ch ^ 1) * ATT_M + r];
      float o[DH];
      if (ok) {
        tc_fence_after();
        load_o<DH>(tO + lane_off + ch * DH, o);
      } else {
#pragma unroll
        for (int e = 0; e < DH; ++e) o[e] = 0.f;
      }
      if (p.splits == 1) {
        if (ok && active) store_out_half<D>(p.out, p.n_max, p.Hq, p.g, b, kvh, pidx, ch, o, 1.f / l_row);
      } else {
        // this split's partial for the merge (the row's (m, l) by half 0)
        float4 *dp = split_slot<D>(p, b, kvh, mtile, split);
#pragma unroll
        for (int c = 0; c < DH; c += 4)
          dp[((ch * DH + c) >> 2) * ATT_M + r] = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
        if (ch == 0) dp[(D / 4) * ATT_M + r] = make_float4(ok ? m_run : -CUDART_INF_F, ok ? l_row : 0.f, 0.f, 0.f);
      }
      if (tid == 0) BST_TRACE_AT(28);
    }
  } else if (p.splits > 1 && tid < ATT_M) {
    // nothing to attend to in this split: an empty (zero) partial
    float4 *dp = split_slot<D>(p, b, kvh, mtile, split);
#pragma unroll
    for (int c = 0; c < D; c += 4) dp[(c >> 2) * ATT_M + r] = make_float4(0.f, 0.f, 0.f, 0.f);
    dp[(D / 4) * ATT_M + r] = make_float4(-CUDART_INF_F, 0.f, 0.f, 0.f);
  }

  // all roles are done with TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (T > 0 && warp == 0) tmem_dealloc(tbase, 512);
  if (T > 0 && *abort && tid == 0) set_err(p.dev_err, BASTION_DEVERR_TIMEOUT);

  // ---- merge of the KV splits: the cluster barrier (release / acquire)
  // publishes every split's partial, then each CTA merges its rows from L2
  if (p.splits > 1) {
    cluster_sync_all();
    if (tid == 0) BST_TRACE_AT(29);
    switch (p.splits) {
      case 2: merge_splits<D, 2>(p, b, kvh, mtile, split, nb); break;
      case 3: merge_splits<D, 3>(p, b, kvh, mtile, split, nb); break;
      case 4: merge_splits<D, 4>(p, b, kvh, mtile, split, nb); break;
      case 5: merge_splits<D, 5>(p, b, kvh, mtile, split, nb); break;
      case 6: merge_splits<D, 6>(p, b, kvh, mtile, split, nb); break;
      case 7: merge_splits<D, 7>(p, b, kvh, mtile, split, nb); break;
      case 8: merge_splits<D, 8>(p, b, kvh, mtile, split, nb); break;
      case 9: merge_splits<D, 9>(p, b, kvh, mtile, split, nb); break;
      case 10: merge_splits<D, 10>(p, b, kvh, mtile, split, nb); break;
      case 11: merge_splits<D, 11>(p, b, kvh, mtile, split, nb); break;
      case 12: merge_splits<D, 12>(p, b, kvh, mtile, split, nb); break;
      case 13: merge_splits<D, 13>(p, b, kvh, mtile, split, nb); break;
      case 14: merge_splits<D, 14>(p, b, kvh, mtile, split, nb); break;
      case 15: merge_splits<D, 15>(p, b, kvh, mtile, split, nb); break;
      default: merge_splits<D, 16>(p, b, kvh, mtile, split, nb); break;
    }
    if (tid == 0) BST_TRACE_AT(30);
  }
  if (tid == 0) BST_TRACE_AT(31);
}

// ================================================================ paged
// caches: one CTA per SM, the batch's work split evenly (see "the work")

// ---------------------------------------------------------------- the work
// A request b with n_b tree nodes has am_b = ceil(n_b g / 128) M-tiles of
// 128 rows per KV head, and each (request, KV head) has T_b tiles of 128 keys:
// its context tiles, then its tree tiles.  The CTAs form gangs of G =
// max_b am_b: member m of a gang computes M-tile m, and the members of a gang
// walk the same tiles at the same time, so each K/V tile crosses from HBM
// into L2 once and is read there by every M-tile.  The (request, KV head)
// pairs with any tree node, in request then KV head order, concatenate to
// W = sum_b Hkv T_b tiles, cut into NG equal gang ranges: gang q takes
// [W q / NG, W (q + 1) / NG).  A unit -- (request, KV head, M-tile) -- cut
// between gangs is finished by the CTA that stores its last piece (a ticket
// per unit); members whose M-tile a request does not have skip its tiles.
struct AttnReq {
  int nb, L, am, ctx_tiles, T;
};
BST_DEV AttnReq load_req(const PagedParams &p, int b) {
  AttnReq r;
  r.nb = p.n[b];
  const bool valid = r.nb >= 1 && r.nb <= p.n_max;
  int L = p.ctx_len[b];
  L = L < 0 ? 0 : (L > p.cap ? static_cast<int>(p.cap) : L);
  r.L = L;
  r.am = valid ? (r.nb * p.g + ATT_M - 1) / ATT_M : 0;
  r.ctx_tiles = (L + ATT_N - 1) / ATT_N;
  r.T = valid ? r.ctx_tiles + (r.nb + ATT_N - 1) / ATT_N : 0;
  return r;
}

// A position in the concatenated tiles: (request b, KV head kvh), tile t of
// its T_b; this CTA computes M-tile m of it.
struct AttnCursor {
  int b, kvh, m, t;
  AttnReq rq;
  int64_t pos;
};

// From the end of (b, kvh) to the start of the next pair whose request has
// M-tile m (requests without tree nodes have no tiles; pairs without M-tile m
// are skipped whole).  Past the last pair, b == B.
BST_DEV void cursor_next_unit(AttnCursor &c, const PagedParams &p) {
  for (;;) {
    if (++c.kvh >= p.Hkv) {
      c.kvh = 0;
      do {
        if (++c.b >= p.B) return;
        c.rq = load_req(p, c.b);
      } while (c.rq.T == 0);
    }
    if (c.m < c.rq.am) return;
    c.pos += c.rq.T;
  }
}
// The cursor of member m at global tile `pos` (< W) or, if that pair has no
// M-tile m, at the start of the next one that has: the request is the last b
// with pre[b] <= pos (requests without tiles have pre[b] == pre[b + 1]).
BST_DEV void cursor_seek(AttnCursor &c, const PagedParams &p, const int64_t *pre, int64_t pos, int m) {
  int lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= pos)
      lo = mid;
    else
      hi = mid;
  }
  c.b = lo;
  c.m = m;
  c.rq = load_req(p, lo);
  const int64_t off = pos - pre[lo];
  c.kvh = static_cast<int>(off / c.rq.T);
  c.t = static_cast<int>(off - static_cast<int64_t>(c.kvh) * c.rq.T);
  c.pos = pos;
  if (m >= c.rq.am) {
    c.pos += c.rq.T - c.t;
    c.t = 0;
    cursor_next_unit(c, p);
  }
}
// the next tile of this member (the caller stops at the end of its range)
BST_DEV void cursor_next(AttnCursor &c, const PagedParams &p) {
  ++c.pos;
  if (++c.t < c.rq.T) return;
  c.t = 0;
  cursor_next_unit(c, p);
}

// Gang of the partition that holds global tile x: the largest q with
// floor(W q / NG) <= x.
BST_DEV int gang_of(int64_t x, int64_t W, int NG) { return static_cast<int>(((x + 1) * NG + W - 1) / W) - 1; }

// Partial slot s of CTA q: slot 0 holds the piece of the unit that starts at
// or before the CTA's range, slot 1 that of a unit starting inside it (at
// most one of each is cut: the units in between are whole).  (D/4 + 1)
// x 128 float4, column-major by float4 (chunk c of row r at c * 128 + r, so a
// warp's store or load of one chunk is 512 contiguous bytes); the last chunk
// of a row holds (m, l, 0, 0) with m in the log2 domain.
template <int D>
BST_DEV float4 *part_slot(const PagedParams &p, int q, int s) {
  return p.part + (static_cast<int64_t>(q) * 2 + s) * (D / 4 + 1) * ATT_M;
}

// Merge of the pieces of unit (b, kvh, M-tile m), cut between gangs q0..q1
// (run by the softmax threads of the CTA that stored the last piece): O =
// sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k, with a running M over chunks
// of eight pieces whose loads are all issued before any is used.  Piece q was
// stored by member m of gang q, in slot 0 unless the unit starts inside the
// gang's range (slot 1).
template <int D>
BST_DEV void merge_pieces(const PagedParams &p, int b, int kvh, int m, int nb, int64_t U0, int64_t W, int NG, int G,
                          int q0, int q1) {
  constexpr int DH = D / 2;
  constexpr int CH = 8;
  const int r = threadIdx.x & (ATT_M - 1);
  const int ch = threadIdx.x >> 7;
  const int row = m * ATT_M + r;
  if (row / p.g >= nb) return;
  float M = -CUDART_INF_F;
  float lsum = 0.f;
  float acc[DH];
#pragma unroll
  for (int c = 0; c < DH; ++c) acc[c] = 0.f;
  for (int qb = q0; qb <= q1; qb += CH) {
    const float4 *src[CH];
    float4 ml[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int q = qb + k;
      src[k] = nullptr;
      ml[k] = make_float4(-CUDART_INF_F, 0.f, 0.f, 0.f);
      if (q <= q1) {
        const int64_t lo_q = (W * q) / NG;
        src[k] = part_slot<D>(p, q * G + m, lo_q >= U0 ? 0 : 1);
        ml[k] = __ldcg(src[k] + (D / 4) * ATT_M + r);
      }
    }
    float Mc = M;
#pragma unroll
    for (int k = 0; k < CH; ++k) Mc = fmaxf(Mc, ml[k].x);
    // earlier chunks' sums to the new reference (pieces that saw no key carry
    // m = -inf, l = 0 and a zero O)
    const float sc = (M == -CUDART_INF_F) ? 0.f : ex2(M - Mc);
    lsum *= sc;
#pragma unroll
    for (int c = 0; c < DH; ++c) acc[c] *= sc;
    float w[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      w[k] = (ml[k].x == -CUDART_INF_F) ? 0.f : ex2(ml[k].x - Mc);
      lsum += w[k] * ml[k].y;
    }
#pragma unroll
    for (int c = 0; c < DH; c += 4) {
      float4 v[CH];
#pragma unroll
      for (int k = 0; k < CH; ++k)
        v[k] = src[k] ? __ldcg(src[k] + ((ch * DH + c) >> 2) * ATT_M + r) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        acc[c] += w[k] * v[k].x;
        acc[c + 1] += w[k] * v[k].y;
        acc[c + 2] += w[k] * v[k].z;
        acc[c + 3] += w[k] * v[k].w;
      }
    }
    M = Mc;
  }
  store_out_half<D>(p.out, p.n_max, p.Hq, p.g, b, kvh, row, ch, acc, 1.f / lsum);
}

// bf16 path: one CTA per SM, each streaming its range of the concatenated
// tiles (see "the work" above).  Roles:
//   warp 8      TMA producer: per unit its Q (after the previous unit's last
//               S finished), per tile the K tile (one tile ahead) and the V
//               tile, 128-byte swizzle; paged caches are gathered page by
//               page through a 4-D tensor map, the page ids read one K tile
//               ahead.
//   warp 9      MMA issuer (one thread): S = Q K^T into TMEM (three S
//               buffers), three tiles ahead of O += P V with P read from TMEM
//               (P aliases its S buffer; the tcgen05.mma of one thread execute
//               in issue order, so S(j + 3), issued after P V(j), cannot
//               overwrite P(j) early).  A unit's first P V starts a new O,
//               once the softmax has read the previous unit's.
//   warps 0-7   softmax: warps q and q + 4 own TMEM lanes 32q..32q+31 (M-tile
//               rows), each one half of the columns; they read S, apply the
//               context bound or the ancestor bits, swap half-row maxima,
//               keep the running max / sum in the log2 domain, write P (bf16)
//               to TMEM and rescale O only when a row max grew by more than
//               2^8 (the exact result is the same for any running reference
//               max).  At the end of a unit they store the output, or a
//               partial and take the unit's ticket; the last piece merges.
// Every mbarrier wait is bounded in time; on expiry the CTA records
// BASTION_DEVERR_TIMEOUT, drains what it issued and frees its TMEM.
template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1) tree_attn_paged_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kt,
    const __grid_constant__ CUtensorMap tm_vt, const PagedParams p) {
  using LY = PagedLayout<D>;
  constexpr int KS = LY::KSTAGES;
  constexpr int VS = LY::VSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + LY::Q_OFF;
  PagedBars *bars = reinterpret_cast<PagedBars *>(smem + LY::BAR_OFF);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int cta = blockIdx.x;

  if (tid == 0) BST_TRACE_AT(0);
  // private set-up first (barriers, descriptor prefetch), then the wait for
  // the grid that produced the tree
  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_free, 1);
    mbar_init(&bars->o_free, ATT_SM_THREADS);
    mbar_init(&bars->o_full, 1);
#pragma unroll
    for (int i = 0; i < KS; ++i) mbar_init(&bars->k_full[i], 1), mbar_init(&bars->k_empty[i], 1);
#pragma unroll
    for (int i = 0; i < VS; ++i) mbar_init(&bars->v_full[i], 1), mbar_init(&bars->v_empty[i], 1);
#pragma unroll
    for (int i = 0; i < ATT_SBUF; ++i) mbar_init(&bars->s_full[i], 1), mbar_init(&bars->p_full[i], ATT_SM_THREADS);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->part_done, ATT_SM_THREADS);
    mbar_init(&bars->part_go, 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(&bars->xbar[i], 64);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == ATT_TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_kt);
    tma_prefetch_desc(&tm_vt);
  }
  pdl_wait();
  pdl_trigger();

  // ---- the partition: warp 0 scans the requests' tiles and finds the gang
  // size (every CTA computes the same; CTA 0 reports bad requests), then
  // counts this member's tiles in its gang's range
  if (warp == 0) {
    int64_t run = 0;
    int am_max = 0;
    if (lane == 0) bars->pre[0] = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int64_t cost = 0;
      if (b < p.B) {
        const AttnReq rq = load_req(p, b);
        cost = static_cast<int64_t>(p.Hkv) * rq.T;
        am_max = max(am_max, rq.am);
        if (cta == 0) {
          if (rq.am == 0) set_err(p.dev_err, BASTION_DEVERR_N);
          const int L = p.ctx_len[b];
          if (L < 0 || L > p.cap) set_err(p.dev_err, BASTION_DEVERR_CTX);
        }
      }
      int64_t x = cost;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
      }
      if (b < p.B) bars->pre[b + 1] = run + x;
      run += __shfl_sync(FULL, x, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am_max = max(am_max, __shfl_xor_sync(FULL, am_max, o));
    if (lane == 0) {
      const int64_t Wt = run;
      const int G = max(am_max, 1);
      // gangs: as many as the grid holds, but at least ATT_MIN_SHARE tiles
      // each (fewer pieces to merge per unit)
      int NG = p.nctas / G;
      const int64_t by_share = (Wt + ATT_MIN_SHARE - 1) / ATT_MIN_SHARE;
      if (by_share < NG) NG = static_cast<int>(by_share);
      if (NG < 1) NG = 1;
      const int q = cta / G;
      int64_t count = 0;
      if (Wt > 0 && q < NG) {
        const int64_t lo = (Wt * q) / NG;
        const int64_t hi = (Wt * (q + 1)) / NG;
        AttnCursor c;
        cursor_seek(c, p, bars->pre, lo, cta - q * G);
        while (c.b < p.B && c.pos < hi) {
          const int64_t e = min(hi, c.pos - c.t + c.rq.T);
          count += e - c.pos;
          if (e == hi) break;
          c.pos = e;
          c.t = 0;
          cursor_next_unit(c, p);
        }
      }
      bars->gang_g = G;
      bars->gang_n = NG;
      bars->my_tiles = static_cast<int>(count);
    }
  }
  __syncthreads();
  const int64_t W = bars->pre[p.B];
  const int G = bars->gang_g;
  const int NG = bars->gang_n;
  const int T = bars->my_tiles;              // tiles of this CTA
  if (T <= 0) return;                        // uniform over the CTA
  const int gang = cta / G;
  const int member = cta - gang * G;
  const int64_t lo = (W * gang) / NG;

  float m_run = -CUDART_INF_F;
  float l_run = 0.f;
  bool ok = true;
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) BST_TRACE_AT(1);
  const uint32_t tbase = bars->tmem_base;
  const uint32_t tO = tbase + ATT_SBUF * 128;

  if (warp == ATT_TMA_WARP) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      BST_TRACE_AT(2);
      constexpr int MAXPG = ATT_N / 8;          // page_size >= 8
      constexpr int PG_BEYOND = -2147483647 - 1;   // token past the context: read zeros
      // page ids of the tile at cursor c
      auto fetch_pages = [&](const AttnCursor &c, bool valid, int (&pg)[MAXPG]) {
        const int ps = p.page_size;
#pragma unroll
        for (int pi = 0; pi < MAXPG; ++pi) {
          const int tok = c.t * ATT_N + pi * ps;
          pg[pi] = (valid && c.t < c.rq.ctx_tiles && pi * ps < ATT_N && tok < c.rq.L)
                       ? __ldg(p.block_table + static_cast<int64_t>(c.b) * p.max_pages + tok / ps)
                       : PG_BEYOND;
        }
      };
      // one K or V tile (context or tree) at cursor c into `dst`, completing
      // on `fb`; pg: the tile's page ids (context tiles)
      auto load_tile = [&](const AttnCursor &c, bool is_v, uint8_t *dst, uint64_t *fb, const int (&pg)[MAXPG]) {
        const CUtensorMap *mc = is_v ? &tm_v : &tm_k;
        const CUtensorMap *mt = is_v ? &tm_vt : &tm_kt;
        if (c.t < c.rq.ctx_tiles) {
          const int ps = p.page_size;
#pragma unroll
          for (int pi = 0; pi < MAXPG; ++pi) {
            if (pi * ps >= ATT_N) break;
            int page = pg[pi];
            if (page == PG_BEYOND) {
              page = p.num_pages;   // out of range: the copy reads zeros
            } else if (page < 0 || page >= p.num_pages) {
              set_err(p.dev_err, BASTION_DEVERR_PAGE);
              page = p.num_pages;
            }
#pragma unroll
            for (int h = 0; h < LY::NH; ++h) tma_load_4d(dst + h * ATT_HALF + pi * ps * 128, mc, fb, h * 64, 0, c.kvh, page);
          }
        } else {
          const int tt = c.t - c.rq.ctx_tiles;
#pragma unroll
          for (int h = 0; h < LY::NH; ++h) tma_load_3d(dst + h * ATT_HALF, mt, fb, h * 64, c.kvh, c.b * p.n_max + tt * ATT_N);
        }
      };
      // K (with Q at the start of each unit) runs one tile ahead of V; the
      // page ids of a K tile are read one K tile before its copy
      AttnCursor ck, cn, cv;
      cursor_seek(ck, p, bars->pre, lo, member);
      cv = ck;
      cn = ck;
      int pgA[MAXPG], pgB[MAXPG], pgN[MAXPG];
      fetch_pages(cn, true, pgN);
      int k_issued = 0, v_issued = 0, units = 0;
      bool run = true;
      auto issue_k = [&](int j) -> bool {
        if (j == 0 || ck.t == 0) {
          // a new unit: its Q, once the previous unit's last S finished
          if (units > 0 && !mbar_wait(&bars->q_free, (units - 1) & 1, abort, ATT_WAIT_NS)) return false;
          mbar_expect_tx(&bars->q_full, LY::Q_BYTES);
#pragma unroll
          for (int h = 0; h < LY::NH; ++h)
            tma_load_3d(sQ + h * ATT_HALF, &tm_q, &bars->q_full, h * 64, ck.kvh * p.g,
                        ck.b * p.n_max + ck.m * (ATT_M / p.g));
          ++units;
        }
        const int st = j % KS;
        // the stage is free once S(j - KS), which read it, is complete
        if (j >= KS && !mbar_wait(&bars->k_empty[st], ((j / KS) - 1) & 1, abort, ATT_WAIT_NS)) return false;
        mbar_expect_tx(&bars->k_full[st], LY::KV_BYTES);
#pragma unroll
        for (int pi = 0; pi < MAXPG; ++pi) {
          pgA[pi] = pgB[pi];
          pgB[pi] = pgN[pi];
        }
        if (j + 1 < T) {
          cursor_next(cn, p);
          fetch_pages(cn, true, pgN);
        }
        load_tile(ck, false, smem + LY::K_OFF + st * LY::KV_BYTES, &bars->k_full[st], pgB);
        if (j < 8) BST_TRACE_AT(32 + j);
        k_issued = j + 1;
        if (j + 1 < T) cursor_next(ck, p);
        return true;
      };
      auto issue_v = [&](int j) -> bool {
        const int st = j % VS;
        if (j >= VS && !mbar_wait(&bars->v_empty[st], ((j / VS) - 1) & 1, abort, ATT_WAIT_NS)) return false;
        mbar_expect_tx(&bars->v_full[st], LY::KV_BYTES);
        // V(j) follows K(j + 1) unless j is the last tile
        load_tile(cv, true, smem + LY::V_OFF + st * LY::KV_BYTES, &bars->v_full[st], j + 1 < T ? pgA : pgB);
        if (j < 8) BST_TRACE_AT(48 + j);
        v_issued = j + 1;
        if (j + 1 < T) cursor_next(cv, p);
        return true;
      };
      run = issue_k(0);
      for (int j = 0; run && j < T; ++j) {
        if (j + 1 < T && !issue_k(j + 1)) break;
        if (!issue_v(j)) break;
      }
      if (*abort) {
        // let the copies already in flight land before the CTA goes away
        for (int j = max(0, k_issued - KS); j < k_issued; ++j)
          mbar_wait(&bars->k_full[j % KS], (j / KS) & 1, abort, ATT_WAIT_NS);
        for (int j = max(0, v_issued - VS); j < v_issued; ++j)
          mbar_wait(&bars->v_full[j % VS], (j / VS) & 1, abort, ATT_WAIT_NS);
        if (units > 0) mbar_wait(&bars->q_full, (units - 1) & 1, abort, ATT_WAIT_NS);
      }
    }
  } else if (warp == ATT_MMA_WARP) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(ATT_M, ATT_N, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16(ATT_M, D, 1);
      // shared-memory descriptors at the bases of Q, K stage 0 and V stage 0
      // (smem addresses stay below 256 KB, so adding (offset >> 4) to a base
      // never carries out of the 14-bit address field)
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(smem + LY::K_OFF), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(smem + LY::V_OFF), ATT_HALF, 1024);
      bool any = false;
      AttnCursor cq, cp;
      cursor_seek(cq, p, bars->pre, lo, member);
      cp = cq;
      int q_units = 0, p_units = 0;
      // S(jj) = Q K(jj)^T into S buffer jj mod 3: one commit tells the softmax
      // that S is ready, one the producer that K stage jj mod KS is free;
      // after a unit's last S a third frees Q
      auto issue_qk = [&](int jj) -> bool {
        if (jj == 0 || cq.t == 0) {
          if (!mbar_wait(&bars->q_full, q_units & 1, abort, ATT_WAIT_NS)) return false;
          ++q_units;
        }
        const int ks = jj % KS;
        const int sb = jj % ATT_SBUF;
        if (!mbar_wait(&bars->k_full[ks], (jj / KS) & 1, abort, ATT_WAIT_NS)) return false;
        if (jj < 8) BST_TRACE_AT(40 + jj);
        tc_fence_after();
        // a descriptor's start address is its low 14 bits (address >> 4), so
        // the K-steps' descriptors are the stage's base plus constants
        const uint64_t kdesc = kdesc0 + static_cast<uint64_t>((ks * LY::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * ATT_HALF + (kk & 3) * 32) >> 4);
          mma_ss(tbase + sb * 128, qdesc0 + off, kdesc + off, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        any = true;
        mma_commit(&bars->s_full[sb]);
        mma_commit(&bars->k_empty[ks]);
        if (jj + 1 == T || cq.t + 1 == cq.rq.T) mma_commit(&bars->q_free);   // the unit's last S
        BST_TRACE_AT(3 + min(jj, 7));
        if (jj + 1 < T) cursor_next(cq, p);
        return true;
      };
      // O += P(jj) V(jj) (a unit's first P V starts a new O, once the softmax
      // has read the previous unit's); one commit frees the V stage and tells
      // the softmax that O holds P(jj) V(jj), another after a unit's last P V
      // that O is final
      auto issue_pv = [&](int jj) -> bool {
        const bool first = (jj == 0 || cp.t == 0);
        if (first) {
          if (p_units > 0 && !mbar_wait(&bars->o_free, (p_units - 1) & 1, abort, ATT_WAIT_NS)) return false;
          ++p_units;
        }
        const int sb = jj % ATT_SBUF;
        const int vs = jj % VS;
        if (!mbar_wait(&bars->p_full[sb], (jj / ATT_SBUF) & 1, abort, ATT_WAIT_NS)) return false;
        if (!mbar_wait(&bars->v_full[vs], (jj / VS) & 1, abort, ATT_WAIT_NS)) return false;
        if (jj < 8) BST_TRACE_AT(56 + jj);
        tc_fence_after();
        // V is the MN-major B operand: 8 keys per 1024-byte swizzle group, the
        // two 64-column halves of d ATT_HALF bytes apart
        const uint64_t vdesc = vdesc0 + static_cast<uint64_t>((vs * LY::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < ATT_N / 16; ++kk)
          mma_ts(tO, tbase + sb * 128 + kk * 8, vdesc + static_cast<uint64_t>((kk * 2048) >> 4), IDESC_PV,
                 (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bars->v_empty[vs]);
        if (jj + 1 == T || cp.t + 1 == cp.rq.T) mma_commit(&bars->o_full);   // the unit's last P V
        if (jj + 1 < T) cursor_next(cp, p);
        return true;
      };
      // S runs three tiles ahead of P V, so the tensor pipe has work queued
      // while the softmax turns S(j) into P(j)
      bool run = true;
      for (int j = 0; run && j < min(T, ATT_SBUF); ++j) run = issue_qk(j);
      for (int j = 0; run && j < T; ++j) {
        if (!issue_pv(j)) { run = false; break; }
        if (j + ATT_SBUF < T && !issue_qk(j + ATT_SBUF)) { run = false; break; }
      }
      if (any) {
        // every MMA issued above has finished before TMEM is released
        mma_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, abort, ATT_WAIT_NS);
      }
    }
  } else {
    // ------------------------------------------------ softmax warps 0-7
    // Warp w owns TMEM lanes 32 (w mod 4) .. +31 (rows) and column half
    // ch = w / 4: keys [64 ch, 64 ch + 64) of every S tile, P columns
    // [32 ch, 32 ch + 32), O columns [D/2 ch, D/2 ch + D/2).  Two warps per
    // scheduler hide each other's TMEM and MUFU latency.
    constexpr int HC = ATT_N / 2;    // S columns per warp
    constexpr int DH = D / 2;        // O columns per warp
    const int rq = warp & 3;
    const int ch = warp >> 2;
    const int r = tid & (ATT_M - 1);
    const uint32_t lane_off = static_cast<uint32_t>(rq * 32) << 16;
    const int W64 = (p.n_max + 63) >> 6;
    const float cs = p.scale_log2;
    uint64_t *xb = &bars->xbar[rq];
    uint32_t xphase = 0;     // swaps through xb so far
    int nparts = 0;          // partials stored so far (part_done / part_go phases)
    int units_done = 0;      // units finished so far (o_full phases)
    int64_t seg0 = lo;       // global index of the current unit's first tile in this CTA
    unsigned long long mw[4] = {0ull, 0ull, 0ull, 0ull};
    AttnCursor c;
    cursor_seek(c, p, bars->pre, lo, member);
    for (int j = 0; j < T; ++j) {
      const bool first = (j == 0 || c.t == 0);
      const bool last = (j + 1 == T || c.t + 1 == c.rq.T);
      const int row = c.m * ATT_M + r;
      const int node = row / p.g;
      if (first) {
        // a new unit: fresh running max / sum, the rows' ancestor bits
        m_run = -CUDART_INF_F;
        l_run = 0.f;
        seg0 = c.pos;
#pragma unroll
        for (int w = 0; w < 4; ++w) mw[w] = 0ull;
        if (node < c.rq.nb) {
          const unsigned long long *mrow = p.mask + (static_cast<int64_t>(c.b) * p.n_max + node) * W64;
          for (int w = 0; w < W64; ++w) mw[w] = mrow[w];
        }
      }
      const int sb = j % ATT_SBUF;
      if (!warp_wait(&bars->s_full[sb], (j / ATT_SBUF) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      if (tid == 0) BST_TRACE_AT(11 + min(j, 7));
      const uint32_t scol = tbase + lane_off + sb * 128 + ch * HC;
      uint32_t s[HC];
      tmem_ld32(scol + 0, s + 0);
      tmem_ld32(scol + 32, s + 32);
      tmem_wait_ld32(s + 0);
      tmem_wait_ld32(s + 32);
      // masking on the raw scores: context tiles are bounded by L, tree
      // tiles by the ancestor bits (masked scores become -inf)
      const uint32_t NEG = 0xff800000u;
      if (c.t < c.rq.ctx_tiles) {
        const int nvalid = c.rq.L - c.t * ATT_N - ch * HC;
        if (nvalid < HC) {
#pragma unroll
          for (int cc = 0; cc < HC; ++cc) s[cc] = (cc < nvalid) ? s[cc] : NEG;
        }
      } else {
        const int tt = c.t - c.rq.ctx_tiles;
        const unsigned long long wb = mw[2 * tt + ch];
#pragma unroll
        for (int cc = 0; cc < HC; ++cc) s[cc] = ((wb >> cc) & 1ull) ? s[cc] : NEG;
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
      for (int cc = 8; cc < HC; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], __uint_as_float(s[cc]));
      const float hmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // swap half maxima with the partner warp; the arrival also tells it
      // this warp's TMEM loads of S are complete (its P stores may then
      // overwrite those columns)
      bars->xmax[xphase & 1][ch][r] = hmax;
      tc_fence_before();
      mbar_arrive(xb);
      if (!warp_wait(xb, xphase & 1, abort)) { ok = false; break; }
      tc_fence_after();
      const float tmax = fmaxf(hmax, bars->xmax[xphase & 1][ch ^ 1][r]) * cs;
      ++xphase;
      const float m_new = fmaxf(m_run, tmax);
      // keep the running reference unless the max grew by more than 2^8
      const bool jump = m_new > m_run + ATT_RESCALE_LOG2;
      const float m_use = jump ? m_new : m_run;
      const float alpha = jump ? ex2(m_run - m_new) : 1.f;
      const float msub = (m_use == -CUDART_INF_F) ? 0.f : m_use;
      float sum[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sum[i] = 0.f;
      uint32_t pk[HC / 2];
#pragma unroll
      for (int cc = 0; cc < HC; cc += 2) {
        const float p0 = ex2(fmaf(__uint_as_float(s[cc]), cs, -msub));
        const float p1 = ex2(fmaf(__uint_as_float(s[cc + 1]), cs, -msub));
        sum[(cc >> 1) & 7] += p0 + p1;
        pk[cc >> 1] = pack_bf16x2(p0, p1);
      }
      tmem_st32(tbase + lane_off + sb * 128 + ch * (HC / 2), pk);
      l_run = l_run * alpha + (((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7])));
      const bool need = !first && jump && (m_run > -CUDART_INF_F);
      if (__any_sync(FULL, need)) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled (the commit after
        // that P V arrives on its V stage's barrier; that barrier is at most
        // one phase behind: S(j) is complete, so P V(j - 3) and every earlier
        // MMA are too)
        if (!warp_wait(&bars->v_empty[(j - 1) % VS], ((j - 1) / VS) & 1, abort)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < DH / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + ch * DH + cc * 32, o);
          tmem_wait_ld32(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + lane_off + ch * DH + cc * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[sb]);
      if (tid == 0) BST_TRACE_AT(19 + min(j, 7));
      m_run = m_use;

      if (last) {
        // ---- end of this CTA's part of the unit: O after its last P V (one
        // o_full phase per unit: unlike a V stage's barrier it cannot be two
        // phases behind), the two halves' row sums added
        if (!warp_wait(&bars->o_full, units_done & 1, abort)) { ok = false; break; }
        ++units_done;
        bars->xl[ch][r] = l_run;
        mbar_arrive(xb);
        if (!warp_wait(xb, xphase & 1, abort)) { ok = false; break; }
        ++xphase;
        const float l_row = l_run + bars->xl[ch ^ 1][r];
        float o[DH];
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < DH / 32; ++cc) {
          uint32_t t32[32];
          tmem_ld32(tO + lane_off + ch * DH + cc * 32, t32);
          tmem_wait_ld32(t32);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[cc * 32 + e] = __uint_as_float(t32[e]);
        }
        // O is in registers: the next unit's first P V may overwrite it
        tc_fence_before();
        mbar_arrive(&bars->o_free);
        const int64_t U0 = c.pos - c.t;   // the unit's first tile
        const bool whole = (seg0 == U0) && (c.t + 1 == c.rq.T);
        if (whole) {
          if (node < c.rq.nb) store_out_half<D>(p.out, p.n_max, p.Hq, p.g, c.b, c.kvh, row, ch, o, 1.f / l_row);
        } else {
          // this CTA's piece of the unit: store it, take the unit's ticket; the
          // CTA that stores the last piece merges them
          float4 *dp = part_slot<D>(p, cta, U0 <= lo ? 0 : 1);
#pragma unroll
          for (int cc = 0; cc < DH; cc += 4)
            dp[((ch * DH + cc) >> 2) * ATT_M + r] = make_float4(o[cc], o[cc + 1], o[cc + 2], o[cc + 3]);
          if (ch == 0) dp[(D / 4) * ATT_M + r] = make_float4(m_run, l_row, 0.f, 0.f);
          __threadfence();
          mbar_arrive(&bars->part_done);
          const int q0 = gang_of(U0, W, NG);
          const int q1 = gang_of(U0 + c.rq.T - 1, W, NG);
          if (tid == 0) {
            int last_piece = 0;
            if (mbar_wait(&bars->part_done, nparts & 1, abort, ATT_WAIT_NS)) {
              uint32_t *tk = p.tickets + (static_cast<int64_t>(c.b) * p.Hkv + c.kvh) * p.mt_max + c.m;
              const uint32_t prev = atomic_add_acq_rel_gpu(tk, 1u);
              last_piece = (prev == static_cast<uint32_t>(q1 - q0)) ? 1 : 0;
              if (last_piece) *tk = 0u;   // every piece is in: the ticket is free for the next call
            }
            bars->last_piece = last_piece;
            mbar_arrive(&bars->part_go);
          }
          if (!warp_wait(&bars->part_go, nparts & 1, abort)) { ok = false; break; }
          ++nparts;
          if (bars->last_piece) {
            __threadfence();
            merge_pieces<D>(p, c.b, c.kvh, c.m, c.rq.nb, U0, W, NG, G, q0, q1);
          }
        }
      }
      if (j + 1 < T) cursor_next(c, p);
    }
    if (tid == 0) BST_TRACE_AT(28);
  }

  // all roles are done with TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
  if (*abort && tid == 0) set_err(p.dev_err, BASTION_DEVERR_TIMEOUT);
  if (tid == 0) BST_TRACE_AT(31);
}

// ------------------------------------------------------------------ fp32 path
struct AttnParamsF32 {
  int n_max, Hq, Hkv, g, d;
  float scale;
  int paged, page_size, max_pages, num_pages;
  int64_t L_max, cap;
  const int32_t *ctx_len;
  const int32_t *n;
  const unsigned long long *mask;
  const int32_t *block_table;
  uint32_t *dev_err;
};

__device__ __forceinline__ const float *f32_ctx_row(const float *base, const AttnParamsF32 &p, int b, int kvh, int j,
                                                    bool *ok) {
  if (!p.paged) return base + ((static_cast<int64_t>(b) * p.Hkv + kvh) * p.L_max + j) * p.d;
  const int page = p.block_table[static_cast<int64_t>(b) * p.max_pages + j / p.page_size];
  if (page < 0 || page >= p.num_pages) {
    *ok = false;
    return base;
  }
  return base + ((static_cast<int64_t>(page) * p.Hkv + kvh) * p.page_size + (j % p.page_size)) * p.d;
}

// One CTA per (head, node, request): 128-key blocks of the context and then of
// the tree are staged in shared memory with coalesced loads (K padded by one
// float per row against bank conflicts), thread t scores key t, and thread e
// accumulates output element e over the block's keys (online softmax, fp32).
constexpr int F32_KEYS = 128;
__host__ __device__ constexpr int f32_smem_bytes(int d) {
  return (F32_KEYS * (d + 1) + F32_KEYS * d) * 4 + F32_KEYS * 8 * 2 + F32_KEYS * 4;
}

__global__ void __launch_bounds__(128) tree_attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ kt,
                                                            const float *__restrict__ vt, const float *__restrict__ kc,
                                                            const float *__restrict__ vc, float *__restrict__ out,
                                                            const AttnParamsF32 p) {
  extern __shared__ __align__(16) float f32s[];
  const int d = p.d;
  float *Ks = f32s;                                   // [F32_KEYS][d + 1]
  float *Vs = Ks + F32_KEYS * (d + 1);                // [F32_KEYS][d]
  const float **kp = reinterpret_cast<const float **>(Vs + F32_KEYS * d);   // row pointers (NULL: no row)
  const float **vp = kp + F32_KEYS;
  float *ps = reinterpret_cast<float *>(vp + F32_KEYS);
  __shared__ float qs[128];
  __shared__ float red[4];
  const int h = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int nb = p.n[b];
  if (nb < 1 || nb > p.n_max) {
    if (tid == 0 && h == 0 && i == 0) set_err(p.dev_err, BASTION_DEVERR_N);
    return;
  }
  if (i >= nb) return;
  int L = p.ctx_len[b];
  if (L < 0 || L > p.cap) {
    if (tid == 0 && h == 0 && i == 0) set_err(p.dev_err, BASTION_DEVERR_CTX);
    L = L < 0 ? 0 : static_cast<int>(p.cap);
  }
  const int kvh = h / p.g;
  const int W = (p.n_max + 63) >> 6;
  const unsigned long long *mrow = p.mask + (static_cast<int64_t>(b) * p.n_max + i) * W;
  if (tid < d) qs[tid] = q[((static_cast<int64_t>(b) * p.n_max + i) * p.Hq + h) * d + tid];
  float m = -CUDART_INF_F, l = 0.f, acc = 0.f;
  const int total = L + nb;
  for (int base = 0; base < total; base += F32_KEYS) {
    const int cnt = min(F32_KEYS, total - base);
    // row pointers of this block's keys; a key is visible when it is a
    // context key with a valid page or an ancestor (or self) in the tree
    {
      const int j = base + tid;
      const float *kr = nullptr, *vr = nullptr;
      if (j < L) {
        bool okp = true;
        kr = f32_ctx_row(kc, p, b, kvh, j, &okp);
        vr = f32_ctx_row(vc, p, b, kvh, j, &okp);
        if (!okp) {
          set_err(p.dev_err, BASTION_DEVERR_PAGE);
          kr = vr = nullptr;
        }
      } else if (j < total) {
        const int jt = j - L;
        if ((mrow[jt >> 6] >> (jt & 63)) & 1ull) {
          kr = kt + ((static_cast<int64_t>(b) * p.n_max + jt) * p.Hkv + kvh) * d;
          vr = vt + ((static_cast<int64_t>(b) * p.n_max + jt) * p.Hkv + kvh) * d;
        }
      }
      kp[tid] = kr;
      vp[tid] = vr;
    }
    __syncthreads();
    // coalesced staging, 16 bytes per load: consecutive threads take
    // consecutive float4 of a row; eight loads in flight per thread before the
    // stores (rows are d floats, d a multiple of 4, bases 16-byte aligned)
    const int d4 = d >> 2;
    for (int i0 = tid; i0 < cnt * d4; i0 += 128 * 8) {
      float4 kv[8], vv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = i0 + u * 128;
        kv[u] = vv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < cnt * d4) {
          const int row = idx / d4, c = idx - row * d4;
          const float *kr = kp[row];
          if (kr) {
            kv[u] = reinterpret_cast<const float4 *>(kr)[c];
            vv[u] = reinterpret_cast<const float4 *>(vp[row])[c];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = i0 + u * 128;
        if (idx < cnt * d4) {
          const int row = idx / d4, c = idx - row * d4;
          float *kd = Ks + row * (d + 1) + 4 * c;
          kd[0] = kv[u].x;
          kd[1] = kv[u].y;
          kd[2] = kv[u].z;
          kd[3] = kv[u].w;
          reinterpret_cast<float4 *>(Vs + row * d)[c] = vv[u];
        }
      }
    }
    __syncthreads();
    float s = -CUDART_INF_F;
    if (tid < cnt && kp[tid]) {
      float a = 0.f;
      const float *kr = Ks + tid * (d + 1);
      for (int e = 0; e < d; ++e) a = fmaf(qs[e], kr[e], a);
      s = a * p.scale;
    }
    float cm = warp_max_f(s);
    if ((tid & 31) == 0) red[tid >> 5] = cm;
    __syncthreads();
    cm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const float m_new = fmaxf(m, cm);
    if (m_new != -CUDART_INF_F) {   // uniform: something is visible
      const float alpha = expf(m - m_new);
      const float pj = (s == -CUDART_INF_F) ? 0.f : expf(s - m_new);
      ps[tid] = pj;
      float cs = warp_sum_f(pj);
      if ((tid & 31) == 0) red[tid >> 5] = cs;
      __syncthreads();
      cs = red[0] + red[1] + red[2] + red[3];
      l = l * alpha + cs;
      acc *= alpha;
      if (tid < d) {
#pragma unroll 8
        for (int jj = 0; jj < cnt; ++jj) acc = fmaf(ps[jj], Vs[jj * d + tid], acc);
      }
      m = m_new;
    }
    __syncthreads();
  }
  if (tid < d) out[((static_cast<int64_t>(b) * p.n_max + i) * p.Hq + h) * d + tid] = acc / l;
}

// ------------------------------------------------------------------ host side
struct AttnPlan {
  int paged;       // 1: the balanced kernel (paged caches), 0: the split kernel
  int mtiles;      // 128-row M-tiles of a (request, KV head) at n_max
  int splits;      // split kernel: KV splits per (request, KV head, M-tile)
  int nctas;       // paged kernel: CTAs (one per SM)
  int64_t cap;
  size_t ws_bytes, ticket_bytes;
};

template <int D>
static int split_smem() { return SplitLayout<D>::SMEM; }

// Clusters of `splits` CTAs of the split kernel that the current device keeps
// resident at once (cached per device, head_dim and cluster size).
static int max_active_clusters(int d, int splits) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, d, splits);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, splits, 1);
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = d == 128 ? split_smem<128>() : split_smem<64>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void *fn = d == 128 ? reinterpret_cast<const void *>(tree_attn_split_kernel<128>)
                            : reinterpret_cast<const void *>(tree_attn_split_kernel<64>);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

AttnPlan plan_tree_attn(int B, int n_max, int Hq, int Hkv, int d, int64_t cap, int num_sms, bool paged) {
  AttnPlan pl{};
  const int g = Hq / Hkv;
  pl.mtiles = (n_max * g + ATT_M - 1) / ATT_M;
  pl.cap = cap;
  pl.paged = paged ? 1 : 0;
  if (paged) {
    // A paged batch is ragged by nature (contexts of any length, trees sized
    // by the controller): one CTA per SM takes an equal share of the batch's
    // actual tiles, found on the device.  Workspace: one ticket word per unit,
    // then two partial slots per CTA.
    pl.nctas = num_sms > 0 ? num_sms : 1;
    pl.splits = 1;
    pl.ticket_bytes = (static_cast<size_t>(B) * Hkv * pl.mtiles * sizeof(uint32_t) + 255) / 256 * 256;
    pl.ws_bytes = pl.ticket_bytes + static_cast<size_t>(pl.nctas) * 2 * (d / 4 + 1) * ATT_M * sizeof(float4);
    return pl;
  }
  // Contiguous cache: KV splits per (request, KV head, M-tile), up to a
  // cluster of 16 (non-portable sizes above 8 count only where the device
  // keeps such clusters resident): the count that minimises (waves of
  // resident clusters) x (tiles per CTA + a fixed cost of about four tiles for
  // set-up, first loads and the merge)
  const int64_t ctx_tiles = (cap + ATT_N - 1) / ATT_N;
  const int64_t tree_tiles = (n_max + ATT_N - 1) / ATT_N;
  const int64_t units = static_cast<int64_t>(B) * Hkv * pl.mtiles;
  const int64_t tot_tiles = ctx_tiles + tree_tiles;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= ATT_MAX_SPLITS; ++s) {
    if (s > 1 && tot_tiles < 2LL * s) break;
    const int per_wave = (s == 1) ? num_sms : max_active_clusters(d, s);
    if (per_wave < 1) continue;
    const int64_t waves = (units + per_wave - 1) / per_wave;
    const double cost = static_cast<double>(waves) * ((s > 1 ? 4.0 : 3.0) + (tot_tiles + s - 1) / s);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  pl.splits = best;
  pl.nctas = 0;
  pl.ticket_bytes = 0;
  // one partial slot per (b, kvh, M-tile, split) when the KV is split
  pl.ws_bytes = best > 1 ? static_cast<size_t>(units) * best * (d / 4 + 1) * ATT_M * sizeof(float4) : 0;
  return pl;
}

cudaError_t prepare_tree_attn() {
  cudaError_t e;
  const void *fns[4] = {reinterpret_cast<const void *>(tree_attn_split_kernel<128>),
                        reinterpret_cast<const void *>(tree_attn_split_kernel<64>),
                        reinterpret_cast<const void *>(tree_attn_paged_kernel<128>),
                        reinterpret_cast<const void *>(tree_attn_paged_kernel<64>)};
  const int smem[4] = {split_smem<128>(), split_smem<64>(), PagedLayout<128>::SMEM, PagedLayout<64>::SMEM};
  for (int i = 0; i < 4; ++i) {
    if (i < 2) {
      e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fns[i], cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(tree_attn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, f32_smem_bytes(128));
  if (e != cudaSuccess) return e;
  return prefer_max_shared(tree_attn_f32_kernel);
}

cudaError_t launch_tree_attn_tc(const CUtensorMap *maps, const AttnPlan &pl, int B, int n_max, int Hq, int Hkv, int d,
                                float scale, int page_size, int max_pages, int num_pages, const int32_t *ctx_len,
                                const int32_t *n, const uint64_t *mask, const int32_t *block_table, void *out,
                                void *ws, uint32_t *dev_err, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  if (!pl.paged) {
    SplitParams p{};
    p.B = B;
    p.n_max = n_max;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.mtiles = pl.mtiles;
    p.splits = pl.splits;
    p.scale_log2 = scale * kLog2e;
    p.cap = pl.cap;
    p.ctx_len = ctx_len;
    p.n = n;
    p.mask = reinterpret_cast<const unsigned long long *>(mask);
    p.out = reinterpret_cast<uint16_t *>(out);
    p.part = reinterpret_cast<float4 *>(ws);
    p.dev_err = dev_err;
    cfg.gridDim = dim3(pl.mtiles, pl.splits, B * Hkv);
    cfg.dynamicSmemBytes = d == 128 ? split_smem<128>() : split_smem<64>();
    cfg.numAttrs = fill_launch_attrs(attr, 1, pl.splits);   // the splits of one (b, kvh, M-tile) form a cluster
    if (d == 128)
      return cudaLaunchKernelEx(&cfg, tree_attn_split_kernel<128>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
    return cudaLaunchKernelEx(&cfg, tree_attn_split_kernel<64>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
  }
  PagedParams p{};
  p.B = B;
  p.n_max = n_max;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.mt_max = pl.mtiles;
  p.nctas = pl.nctas;
  p.scale_log2 = scale * kLog2e;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.cap = pl.cap;
  p.ctx_len = ctx_len;
  p.n = n;
  p.mask = reinterpret_cast<const unsigned long long *>(mask);
  p.block_table = block_table;
  p.out = reinterpret_cast<uint16_t *>(out);
  p.tickets = reinterpret_cast<uint32_t *>(ws);
  p.part = reinterpret_cast<float4 *>(reinterpret_cast<char *>(ws) + pl.ticket_bytes);
  p.dev_err = dev_err;
  cfg.gridDim = dim3(pl.nctas, 1, 1);
  cfg.dynamicSmemBytes = d == 128 ? PagedLayout<128>::SMEM : PagedLayout<64>::SMEM;
  cfg.numAttrs = fill_launch_attrs(attr);
  if (d == 128)
    return cudaLaunchKernelEx(&cfg, tree_attn_paged_kernel<128>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cudaLaunchKernelEx(&cfg, tree_attn_paged_kernel<64>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
}

cudaError_t launch_tree_attn_f32(const float *q, const float *kt, const float *vt, const float *kc, const float *vc,
                                 float *out, int B, int n_max, int Hq, int Hkv, int d, float scale, bool paged,
                                 int64_t L_max, int page_size, int max_pages, int num_pages, int64_t cap,
                                 const int32_t *ctx_len, const int32_t *n, const uint64_t *mask,
                                 const int32_t *block_table, uint32_t *dev_err, cudaStream_t stream) {
  AttnParamsF32 p{};
  p.n_max = n_max;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.d = d;
  p.scale = scale;
  p.paged = paged ? 1 : 0;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.L_max = L_max;
  p.cap = cap;
  p.ctx_len = ctx_len;
  p.n = n;
  p.mask = reinterpret_cast<const unsigned long long *>(mask);
  p.block_table = block_table;
  p.dev_err = dev_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Hq, n_max, B);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(f32_smem_bytes(d));
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = fill_launch_attrs(attr);
  return cudaLaunchKernelEx(&cfg, tree_attn_f32_kernel, q, kt, vt, kc, vc, out, p);
}

}  // namespace bst
