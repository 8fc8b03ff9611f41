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
// bf16 path (tcgen05): one CTA per (request b, KV head, 128-row M-tile, KV
// split), or one CTA pair per two M-tiles (see the kernel).  The M rows pack
// g = Hq/Hkv query heads x tree nodes of one KV head (GQA), so every K/V tile
// is used by all heads of its group.  Roles:
//   warp 8      TMA producer: Q once, then K tiles (128 keys, running one
//               tile ahead) and V tiles, in rings, 128-byte swizzle; paged
//               caches are gathered page by page through a 4-D tensor map;
//               no multicast.
//   warp 9      MMA issuer (one thread): S = Q K^T into TMEM (three S
//               buffers, each freed by its own barrier once the P V that
//               read it finished), O += P V with P read from TMEM (P aliases
//               its S buffer).
//   warps 0-7   softmax: warps q and q + 4 own TMEM lanes 32q..32q+31 (M-tile
//               rows), each one half of the columns; they read S, apply the
//               context bound or the ancestor bits, swap half-row maxima,
//               keep the running max / sum in the log2 domain, write P
//               (bf16) to TMEM, and rescale O only when a row max grew by
//               more than 2^8 (the exact result is the same for any running
//               reference max).
// A request's context tiles followed by its tree tiles are spread evenly over
// the KV splits.  The splits of one (b, kvh, M-tile) form one thread-block
// cluster: each CTA stores its partial (O, m, l) to the workspace in L2, one
// cluster barrier publishes them, and every CTA merges a slice of the rows.
// Every mbarrier wait is bounded in time; on expiry the CTA records
// BASTION_DEVERR_TIMEOUT, drains what it issued and frees its TMEM.
//
// f32 path: an exact fp32 flash-decoding kernel, one CTA per (b, node, head),
// 128-key blocks staged in shared memory.
#include <cooperative_groups.h>
#include <math_constants.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace bst {

constexpr int ATT_THREADS = 320;        // 8 softmax warps, a TMA warp, an MMA warp
constexpr int ATT_TMA_WARP = 8;
constexpr int ATT_MMA_WARP = 9;
constexpr int ATT_N = 128;              // keys per tile
constexpr int ATT_M = 128;              // rows per M-tile
constexpr int ATT_HALF = ATT_N * 128;   // bytes of 128 rows x 64 bf16
constexpr int ATT_VSTAGES = 3;         // V ring depth of the single-CTA form (head_dim 64)
constexpr int ATT_MAX_STAGES = 4;      // of either form
constexpr int ATT_SBUF = 3;             // S / P buffers in TMEM (128 columns each; O follows)
constexpr int ATT_MAX_SPLITS = 16;      // cluster size; above 8 (non-portable) where the device keeps them resident
constexpr uint64_t ATT_WAIT_NS = 200ull * 1000ull * 1000ull;
constexpr float ATT_RESCALE_LOG2 = 8.f;

struct AttnParams {
  int B, n_max, Hq, Hkv, g, mtiles, splits, tiles_per_split;
  float scale_log2;          // scale * log2(e)
  int page_size, max_pages, num_pages;
  int64_t cap;               // context capacity per request
  const int32_t *ctx_len;
  const int32_t *n;
  const unsigned long long *mask;
  const int32_t *block_table;
  uint16_t *out;             // bf16 [B, n_max, Hq, d]
  float4 *part;              // split partials (workspace), used when splits > 1
  uint32_t *dev_err;
};

struct AttnBars {
  uint64_t q_full;
  uint64_t k_full[ATT_MAX_STAGES];
  uint64_t v_full[ATT_MAX_STAGES];
  uint64_t v_empty[ATT_MAX_STAGES];   // P V(j) finished (V stage j free, O updated)
  uint64_t s_full[ATT_SBUF];          // S(j) finished (S ready, K stage j mod 3 free)
  uint64_t p_full[ATT_SBUF];
  uint64_t drain;
  // the two softmax warps that share a row quarter (warps q and q + 4, one
  // half of the columns each) swap their row maxima every tile, and their
  // row sums at the end, through xmax / xl; xbar[q] completes once per swap
  uint64_t xbar[4];
  float xmax[2][2][ATT_M];   // [tile parity][column half][row]
  float xl[2][ATT_M];        // [column half][row]
  uint32_t tmem_base;
  int abort;
};

template <int D, bool kPair>
struct AttnLayout {
  static constexpr int NH = D / 64;
  // a CTA pair needs head_dim 128: each CTA holds one 64-column half of V
  static_assert(!kPair || D == 128, "the CTA-pair form needs head_dim 128");
  // K stage j mod 3 is S buffer j mod 3 (one barrier serves both)
  static constexpr int KSTAGES = ATT_SBUF;
  // (a single CTA with head_dim 128 keeps two V tiles: three do not fit next
  // to three K tiles, Q and the barriers)
  static constexpr int VSTAGES = kPair ? 4 : (D == 128 ? 2 : ATT_VSTAGES);
  static constexpr int Q_BYTES = NH * ATT_HALF;
  // one CTA's part of a K tile: 128 keys (alone) or its 64 keys (pair), each
  // as NH column halves of 64 d; of a V tile: every d half (alone) or its one
  // half (pair), 128 keys each
  static constexpr int K_HALF = kPair ? ATT_HALF / 2 : ATT_HALF;
  static constexpr int K_BYTES = NH * K_HALF;
  static constexpr int V_BYTES = kPair ? ATT_HALF : NH * ATT_HALF;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_BYTES;
  static constexpr int V_OFF = K_OFF + KSTAGES * K_BYTES;
  static constexpr int BAR_OFF = V_OFF + VSTAGES * V_BYTES;

  static constexpr int USED = BAR_OFF + static_cast<int>(sizeof(AttnBars));
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

// KV-split partials live in the workspace, one slot per (b, kvh, M-tile,
// split): (D/4 + 1) x 128 float4, column-major by float4 (chunk c of row r at
// c * 128 + r, so a warp's store or load of one chunk is 512 contiguous
// bytes); the last chunk of a row holds (m, l, 0, 0) with m in the log2 domain.
template <int D>
BST_DEV float4 *part_slot(const AttnParams &p, int b, int kvh, int mtile, int split) {
  const int64_t slot = ((static_cast<int64_t>(b) * p.Hkv + kvh) * p.mtiles + mtile) * p.splits + split;
  return p.part + slot * (D / 4 + 1) * ATT_M;
}

// Merge of the S split partials (every CTA of the cluster, after a cluster
// barrier that follows all main loops and partial stores).  CTA `split` owns
// R = ceil(128 / S) rows of the M-tile: O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s.  G threads share a row, each taking CPG of its D/4
// float4 columns; every load is issued before any is used (one L2 round trip).
template <int D, int S>
BST_DEV void merge_splits(const AttnParams &p, int b, int kvh, int mtile, int split, int nb) {
  constexpr int R = (ATT_M + S - 1) / S;
  constexpr int G = ATT_THREADS / R;
  constexpr int NC4 = D / 4;
  constexpr int CPG = (NC4 + G - 1) / G;
  const int tid = threadIdx.x;
  if (tid >= R * G) return;
  const int rl = tid % R;
  const int rr = split * R + rl;
  if (rr >= ATT_M) return;
  const int g = tid / R;
  const int c40 = g * CPG;
  const int prow = mtile * ATT_M + rr;
  const int nd = prow / p.g;
  if (nd >= nb) return;
  float4 ml[S];
  float4 ov[S][CPG];
#pragma unroll
  for (int s2 = 0; s2 < S; ++s2) {
    const float4 *src = part_slot<D>(p, b, kvh, mtile, s2);
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

// kPair = false: one CTA per (request, KV head, 128-row M-tile, KV split).
// kPair = true: the two M-tiles 2p and 2p+1 of a (request, KV head) run as a
// CTA pair (cta_group::2) on two SMs: each CTA loads its own 128 rows of Q,
// half the keys of every K tile (64 of 128) and one 64-column half of every V
// tile, and the leader (even) CTA issues M = 256 MMAs that read both CTAs'
// shared memory and write both CTAs' TMEM.  Every K/V byte then crosses L2 to
// one SM instead of two, and each SM's shared memory feeds half of the B
// operand.  The pair's copies complete on the leader's barriers; the leader's
// commits arrive on both CTAs' barriers; the peer's softmax warps arrive on
// the leader's P barrier remotely.
template <int D, bool kPaged, bool kPair>
__global__ void __launch_bounds__(ATT_THREADS, 1) tree_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kt,
    const __grid_constant__ CUtensorMap tm_vt, const AttnParams p) {
  using LY = AttnLayout<D, kPair>;
  constexpr int KS = LY::KSTAGES;
  constexpr int VS = LY::VSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + LY::Q_OFF;
  AttnBars *bars = reinterpret_cast<AttnBars *>(smem + LY::BAR_OFF);
  volatile int *abort = &bars->abort;
  cg::cluster_group cluster = cg::this_cluster();

  const int mtile = blockIdx.x;
  const int split = blockIdx.y;   // the cluster spans the splits (blockIdx.y), and the pair (blockIdx.x)
  const int bh = blockIdx.z;
  const int b = bh / p.Hkv;
  const int kvh = bh - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  // CTA pair: the peer CTA's %cluster_ctarank differs in bit 0 (blockIdx.x & 1)
  const uint32_t crank = kPair ? cluster_ctarank() : 0u;
  const uint32_t lead_rank = crank & ~1u;
  const int half = kPair ? (blockIdx.x & 1) : 0;   // which half of each K and V tile this CTA loads
  const bool leader = half == 0;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);

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
    for (int i = 0; i < ATT_SBUF; ++i)   // P: every softmax thread (alone) or one lane per softmax warp of both CTAs
      mbar_init(&bars->s_full[i], 1), mbar_init(&bars->p_full[i], kPair ? 16 : 256);
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
  // no active row in this M-tile (alone) or in the pair's first M-tile (pair:
  // both CTAs take the same exit)
  if ((kPair ? (mtile & ~1) : mtile) * ATT_M >= nb * p.g) return;

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

  // a pair's barriers are initialised before either CTA signals the other's
  if (kPair) cluster_sync_all();
  if (T > 0 && warp == 0) {
    if (kPair) {
      tmem_alloc_pair(&bars->tmem_base, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_base, 512);
      tmem_relinquish();
    }
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
        // a copy completes on this CTA's barrier (alone) or on the leader's
        // (pair: the leader expects both CTAs' bytes)
        auto tma3 = [&](void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1, int c2) {
          if (kPair)
            tma_load_3d_pair(dst, m, mapa_shared(bar, lead_rank), c0, c1, c2);
          else
            tma_load_3d(dst, m, bar, c0, c1, c2);
        };
        auto tma4 = [&](void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1, int c2, int c3) {
          if (kPair)
            tma_load_4d_pair(dst, m, mapa_shared(bar, lead_rank), c0, c1, c2, c3);
          else
            tma_load_4d(dst, m, bar, c0, c1, c2, c3);
        };
        constexpr uint32_t TX_MUL = kPair ? 2u : 1u;
        if (leader) mbar_expect_tx(&bars->q_full, TX_MUL * LY::Q_BYTES);
#pragma unroll
        for (int h = 0; h < LY::NH; ++h)
          tma3(sQ + h * ATT_HALF, &tm_q, &bars->q_full, h * 64, kvh * p.g, b * p.n_max + mtile * (ATT_M / p.g));
        // Paged caches: the page ids of a context tile are read from the block
        // table with all loads in flight together, one K tile ahead of the copy
        // that needs them, so their latency hides behind the previous tile; the
        // V copy of a tile reuses the ids its K copy read.  pgB holds the ids of
        // the last K tile issued, pgA those of the one before, pgN the next.
        constexpr int MAXPG = ATT_N / 8;          // page_size >= 8
        constexpr int PG_BEYOND = -2147483647 - 1;   // token past the context: read zeros
        int pgA[MAXPG], pgB[MAXPG], pgN[MAXPG];
        auto fetch_pages = [&](int j) {
          if (!kPaged) return;
          const int ps = p.page_size;
#pragma unroll
          for (int pi = 0; pi < MAXPG; ++pi) {
            const int tok = (ct0 + j) * ATT_N + pi * ps;
            pgN[pi] = (j < n_ctx && pi * ps < ATT_N && tok < L)
                          ? __ldg(p.block_table + static_cast<int64_t>(b) * p.max_pages + tok / ps)
                          : PG_BEYOND;
          }
        };
        // checked page id (out of range: the copy reads zeros and the error
        // word says so)
        auto page_of = [&](int page) {
          if (page == PG_BEYOND) return p.num_pages;
          if (page < 0 || page >= p.num_pages) {
            set_err(p.dev_err, BASTION_DEVERR_PAGE);
            return p.num_pages;
          }
          return page;
        };
        // This CTA's part of K tile j (context or tree) into `dst`, completing
        // on `fb`: all 128 keys (alone) or keys [64 half, 64 half + 64) (pair),
        // as LY::NH column halves of 64 d.  pg: the tile's page ids.
        auto load_k = [&](int j, uint8_t *dst, uint64_t *fb, const int (&pg)[MAXPG]) {
          const int key0 = kPair ? half * (ATT_N / 2) : 0;
          if (j < n_ctx) {
            const int ct = ct0 + j;
            if (!kPaged) {
#pragma unroll
              for (int h = 0; h < LY::NH; ++h)
                tma3(dst + h * LY::K_HALF, &tm_k, fb, h * 64, ct * ATT_N + key0, b * p.Hkv + kvh);
            } else {
              const int ps = p.page_size;
              const int np = (kPair ? ATT_N / 2 : ATT_N) / ps;   // pages of this CTA's keys
              const int pi0 = key0 / ps;
#pragma unroll
              for (int pj = 0; pj < MAXPG; ++pj) {
                if (pj >= np) break;
                const int page = page_of(pg[pi0 + pj]);
#pragma unroll
                for (int h = 0; h < LY::NH; ++h) tma4(dst + h * LY::K_HALF + pj * ps * 128, &tm_k, fb, h * 64, 0, kvh, page);
              }
            }
          } else {
            const int tt = tr0 + j - n_ctx;
#pragma unroll
            for (int h = 0; h < LY::NH; ++h)
              tma3(dst + h * LY::K_HALF, &tm_kt, fb, h * 64, kvh, b * p.n_max + tt * ATT_N + key0);
          }
        };
        // This CTA's part of V tile j: every d half (alone) or d half `half`
        // (pair), all 128 keys.
        auto load_v = [&](int j, uint8_t *dst, uint64_t *fb, const int (&pg)[MAXPG]) {
          constexpr int NVH = kPair ? 1 : LY::NH;
          if (j < n_ctx) {
            const int ct = ct0 + j;
            if (!kPaged) {
#pragma unroll
              for (int h = 0; h < NVH; ++h)
                tma3(dst + h * ATT_HALF, &tm_v, fb, (h + half) * 64, ct * ATT_N, b * p.Hkv + kvh);
            } else {
              const int ps = p.page_size;
#pragma unroll
              for (int pi = 0; pi < MAXPG; ++pi) {
                if (pi * ps >= ATT_N) break;
                const int page = page_of(pg[pi]);
#pragma unroll
                for (int h = 0; h < NVH; ++h) tma4(dst + h * ATT_HALF + pi * ps * 128, &tm_v, fb, (h + half) * 64, 0, kvh, page);
              }
            }
          } else {
            const int tt = tr0 + j - n_ctx;
#pragma unroll
            for (int h = 0; h < NVH; ++h)
              tma3(dst + h * ATT_HALF, &tm_vt, fb, (h + half) * 64, kvh, b * p.n_max + tt * ATT_N);
          }
        };
        int k_issued = 0, v_issued = 0;
        auto issue_k = [&](int j) -> bool {
          const int st = j % KS;
          // the stage is free once S(j - KS), which read it, is complete
          if (j >= KS && !mbar_wait(&bars->s_full[st], ((j / KS) - 1) & 1, abort, ATT_WAIT_NS)) return false;
          if (leader) mbar_expect_tx(&bars->k_full[st], TX_MUL * LY::K_BYTES);
          if (kPaged) {
#pragma unroll
            for (int pi = 0; pi < MAXPG; ++pi) {
              pgA[pi] = pgB[pi];
              pgB[pi] = pgN[pi];
            }
            fetch_pages(j + 1);
          }
          load_k(j, smem + LY::K_OFF + st * LY::K_BYTES, &bars->k_full[st], pgB);
          if (j < 8) BST_TRACE_AT(32 + j);
          k_issued = j + 1;
          return true;
        };
        auto issue_v = [&](int j) -> bool {
          const int st = j % VS;
          if (j >= VS && !mbar_wait(&bars->v_empty[st], ((j / VS) - 1) & 1, abort, ATT_WAIT_NS)) return false;
          if (leader) mbar_expect_tx(&bars->v_full[st], TX_MUL * LY::V_BYTES);
          // V(j) follows K(j + 1) unless j is the last tile
          load_v(j, smem + LY::V_OFF + st * LY::V_BYTES, &bars->v_full[st], j + 1 < T ? pgA : pgB);
          if (j < 8) BST_TRACE_AT(48 + j);
          v_issued = j + 1;
          return true;
        };
        // K runs one tile ahead of V
        fetch_pages(0);
        bool run = issue_k(0);
        for (int j = 0; run && j < T; ++j) {
          if (j + 1 < T && !issue_k(j + 1)) break;
          if (!issue_v(j)) break;
        }
        if (*abort) {
          // let the copies already in flight land before the CTA goes away
          // (a pair's copies complete on the leader's barriers: the leader
          // waits for both CTAs' bytes; the peer stays until the final
          // cluster barrier)
          if (leader) {
            for (int j = max(0, k_issued - KS); j < k_issued; ++j)
              mbar_wait(&bars->k_full[j % KS], (j / KS) & 1, abort, ATT_WAIT_NS);
            for (int j = max(0, v_issued - VS); j < v_issued; ++j)
              mbar_wait(&bars->v_full[j % VS], (j / VS) & 1, abort, ATT_WAIT_NS);
            mbar_wait(&bars->q_full, 0, abort, ATT_WAIT_NS);
          }
        }
      }
    } else if (warp == ATT_MMA_WARP) {
      // ------------------------------------------------ MMA issuer (the leader of a pair)
      if (lane == 0 && leader) {
        constexpr int MM = kPair ? 2 * ATT_M : ATT_M;
        constexpr uint32_t IDESC_QK = idesc_bf16(MM, ATT_N, 0);
        constexpr uint32_t IDESC_PV = idesc_bf16(MM, D, 1);
        const uint32_t q_addr = smem_u32(sQ);
        auto commit = [&](uint64_t *bar) {
          if (kPair)
            mma_commit_pair(bar, pair_mask);
          else
            mma_commit(bar);
        };
        auto mma_ss_ = [&](uint32_t d_, uint64_t a_, uint64_t b_, uint32_t i_, uint32_t acc) {
          if (kPair)
            mma_ss_pair(d_, a_, b_, i_, acc);
          else
            mma_ss(d_, a_, b_, i_, acc);
        };
        auto mma_ts_ = [&](uint32_t d_, uint32_t a_, uint64_t b_, uint32_t i_, uint32_t acc) {
          if (kPair)
            mma_ts_pair(d_, a_, b_, i_, acc);
          else
            mma_ts(d_, a_, b_, i_, acc);
        };
        bool any = false;
        // S(jj) = Q K(jj)^T into S buffer jj mod 3, which is also K stage
        // jj mod 3: one commit tells the softmax that S is ready and the
        // producer that the K stage is free
        auto issue_qk = [&](int jj) -> bool {
          const int ks = jj % KS;
          if (!mbar_wait(&bars->k_full[ks], (jj / KS) & 1, abort, ATT_WAIT_NS)) return false;
          if (jj < 8) BST_TRACE_AT(40 + jj);
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + LY::K_OFF + ks * LY::K_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int h = kk >> 2;
            const uint64_t adesc = sdesc_sw128(q_addr + h * ATT_HALF + (kk & 3) * 32, 16, 1024);
            const uint64_t bdesc = sdesc_sw128(k_addr + h * LY::K_HALF + (kk & 3) * 32, 16, 1024);
            mma_ss_(tbase + ks * 128, adesc, bdesc, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          any = true;
          commit(&bars->s_full[ks]);
          BST_TRACE_AT(3 + min(jj, 7));
          return true;
        };
        // O += P(jj) V(jj); one commit frees the V stage and tells the softmax
        // that O holds P(jj) V(jj) (before it rescales O)
        auto issue_pv = [&](int jj) -> bool {
          const int sb = jj % ATT_SBUF;
          const int vs = jj % VS;
          // P arrives from this CTA's softmax threads (alone) or from one lane
          // of each softmax warp of both CTAs (pair)
          if (!mbar_wait(&bars->p_full[sb], (jj / ATT_SBUF) & 1, abort, ATT_WAIT_NS)) return false;
          if (!mbar_wait(&bars->v_full[vs], (jj / VS) & 1, abort, ATT_WAIT_NS)) return false;
          if (jj < 8) BST_TRACE_AT(56 + jj);
          tc_fence_after();
          const uint32_t v_addr = smem_u32(smem + LY::V_OFF + vs * LY::V_BYTES);
#pragma unroll
          for (int kk = 0; kk < ATT_N / 16; ++kk) {
            // V is the MN-major B operand: 8 keys per 1024-byte swizzle group;
            // alone, the two 64-column halves of d are ATT_HALF bytes apart;
            // in a pair each CTA holds its one half (N split across the pair)
            const uint64_t bdesc = sdesc_sw128(v_addr + kk * 2048, ATT_HALF, 1024);
            mma_ts_(tO, tbase + sb * 128 + kk * 8, bdesc, IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          commit(&bars->v_empty[vs]);
          return true;
        };
        bool run = mbar_wait(&bars->q_full, 0, abort, ATT_WAIT_NS);
        tc_fence_after();
        // S runs three tiles ahead of P V, so the tensor pipe has work queued
        // while the softmax turns S(j) into P(j).  S(j + 3) reuses the buffer
        // of S(j) / P(j); it is issued after P V(j), which read P(j) there, and
        // the tcgen05.mma of one thread execute in issue order.
        for (int j = 0; run && j < min(T, ATT_SBUF); ++j) run = issue_qk(j);
        for (int j = 0; run && j < T; ++j) {
          if (!issue_pv(j)) { run = false; break; }
          if (j + ATT_SBUF < T && !issue_qk(j + ATT_SBUF)) { run = false; break; }
        }
        if (any) {
          // every MMA issued above has finished before TMEM is released
          commit(&bars->drain);
          mbar_wait(&bars->drain, 0, abort, ATT_WAIT_NS);
        }
      }
    } else {
      // ------------------------------------------------ softmax warps 0-7
      // Warp w owns TMEM lanes 32 (w mod 4) .. +31 (rows) and column half
      // ch = w / 4: keys [64 ch, 64 ch + 64) of every S tile, P columns
      // [32 ch, 32 ch + 32), O columns [D/2 ch, D/2 ch + D/2).  Two warps per
      // scheduler hide each other's TMEM and MUFU latency.  Per tile they
      // swap half-row maxima (so both take the same reference max and
      // rescale decision) and at the end their half-row sums.
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
        const uint32_t scol = tbase + lane_off + sb * 128 + ch * HC;
        uint32_t s[HC];
        tmem_ld32(scol + 0, s + 0);
        tmem_ld32(scol + 32, s + 32);
        tmem_wait_ld32(s + 0);
        tmem_wait_ld32(s + 32);
        // masking on the raw scores: context tiles are bounded by L, tree
        // tiles by the ancestor bits (masked scores become -inf)
        const uint32_t NEG = 0xff800000u;
        if (j < n_ctx) {
          const int nvalid = L - (ct0 + j) * ATT_N - ch * HC;
          if (nvalid < HC) {
#pragma unroll
            for (int c = 0; c < HC; ++c) s[c] = (c < nvalid) ? s[c] : NEG;
          }
        } else {
          const int tt = tr0 + j - n_ctx;
          const unsigned long long wb = mw[2 * tt + ch];
#pragma unroll
          for (int c = 0; c < HC; ++c) s[c] = ((wb >> c) & 1ull) ? s[c] : NEG;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
        for (int c = 8; c < HC; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(s[c]));
        const float hmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
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
        const float msub = (m_use == -CUDART_INF_F) ? 0.f : m_use;
        float sum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) sum[i] = 0.f;
        uint32_t pk[HC / 2];
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(s[c]), cs, -msub));
          const float p1 = ex2(fmaf(__uint_as_float(s[c + 1]), cs, -msub));
          sum[(c >> 1) & 7] += p0 + p1;
          pk[c >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tbase + lane_off + sb * 128 + ch * (HC / 2), pk);
        l_run = l_run * alpha + (((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7])));
        const bool need = (j >= 1) && jump && (m_run > -CUDART_INF_F);
        if (__any_sync(FULL, need)) {
          // O must hold P_{j-1} V_{j-1} before it is rescaled (the commit after
          // that P V arrives on its V stage's barrier)
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
        if (kPair) {
          // one arrival per warp on the leader's barrier, after every lane's
          // TMEM stores completed
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(&bars->p_full[sb], lead_rank));
        } else {
          mbar_arrive(&bars->p_full[sb]);
        }
        if (tid == 0) BST_TRACE_AT(19 + min(j, 7));
        m_run = m_use;
      }
      // ---- epilogue: O after the last P V (the drain barrier completes once,
      // after every MMA of this CTA or pair); the two halves' row sums add
      if (ok && !warp_wait(&bars->drain, 0, abort)) ok = false;
      if (tid == 0) BST_TRACE_AT(27);
      bars->xl[ch][r] = l_run;
      mbar_arrive(xb);
      if (ok && !warp_wait(xb, T & 1, abort)) ok = false;
      const float l_row = l_run + bars->xl[ch ^ 1][r];
      float o[DH];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < DH / 32; ++cc) {
          uint32_t t32[32];
          tmem_ld32(tO + lane_off + ch * DH + cc * 32, t32);
          tmem_wait_ld32(t32);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[cc * 32 + e] = __uint_as_float(t32[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < DH; ++e) o[e] = 0.f;
      }
      if (p.splits == 1) {
        if (ok && active) {
          const float inv = 1.f / l_row;
          const int hl = pidx - node * p.g;
          uint16_t *dst = p.out + ((static_cast<int64_t>(b) * p.n_max + node) * p.Hq + kvh * p.g + hl) * D + ch * DH;
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
      } else {
        // this split's partial for the merge (the row's (m, l) by half 0)
        float4 *dp = part_slot<D>(p, b, kvh, mtile, split);
#pragma unroll
        for (int c = 0; c < DH; c += 4)
          dp[((ch * DH + c) >> 2) * ATT_M + r] = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
        if (ch == 0) dp[(D / 4) * ATT_M + r] = make_float4(ok ? m_run : -CUDART_INF_F, ok ? l_row : 0.f, 0.f, 0.f);
      }
      if (tid == 0) BST_TRACE_AT(28);
    }
  } else if (p.splits > 1 && tid < 128) {
    // nothing to attend to in this split: an empty (zero) partial
    float4 *dp = part_slot<D>(p, b, kvh, mtile, split);
#pragma unroll
    for (int c = 0; c < D; c += 4) dp[(c >> 2) * ATT_M + r] = make_float4(0.f, 0.f, 0.f, 0.f);
    dp[(D / 4) * ATT_M + r] = make_float4(-CUDART_INF_F, 0.f, 0.f, 0.f);
  }

  // all roles are done with TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (kPair && *abort && !leader && tid == 0) {
    // the pair's copies into this CTA complete on the leader's barriers, which
    // this CTA cannot watch: give any still in flight a bounded time to land
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2ull * 1000ull * 1000ull) {
    }
  }
  if (T > 0 && warp == 0) {
    if (kPair)
      tmem_dealloc_pair(tbase, 512);
    else
      tmem_dealloc(tbase, 512);
  }
  if (T > 0 && *abort && tid == 0) set_err(p.dev_err, BASTION_DEVERR_TIMEOUT);

  // ---- merge of the KV splits: the cluster barrier (release / acquire)
  // publishes every split's partial, then each CTA merges its rows from L2.
  // A pair always meets here too: neither CTA leaves while the other may
  // still signal it.
  if (kPair || p.splits > 1) cluster.sync();
  if (p.splits > 1) {
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
  int mtiles, splits, tiles_per_split;
  int pair;   // 1: CTA pairs (cta_group::2) over M-tiles 2p, 2p+1
  int64_t cap;
  size_t ws_bytes, off_o, off_ml;
};

template <bool kPair>
static const void *attn_kernel_fn(int d, bool paged) {
  if (kPair) {
    return paged ? reinterpret_cast<const void *>(tree_attn_tc_kernel<128, true, true>)
                 : reinterpret_cast<const void *>(tree_attn_tc_kernel<128, false, true>);
  }
  return d == 128 ? (paged ? reinterpret_cast<const void *>(tree_attn_tc_kernel<128, true, false>)
                           : reinterpret_cast<const void *>(tree_attn_tc_kernel<128, false, false>))
                  : (paged ? reinterpret_cast<const void *>(tree_attn_tc_kernel<64, true, false>)
                           : reinterpret_cast<const void *>(tree_attn_tc_kernel<64, false, false>));
}

static int attn_smem_bytes(int d, bool pair) {
  if (pair) return AttnLayout<128, true>::SMEM;
  return d == 128 ? AttnLayout<128, false>::SMEM : AttnLayout<64, false>::SMEM;
}

// Clusters of (pair ? 2 : 1) x `splits` CTAs of the bf16 kernel that the
// current device keeps resident at once (cached per device, head_dim, layout,
// form and cluster size).
static int max_active_clusters(int d, bool paged, bool pair, int splits) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, d, paged ? 1 : 0, pair ? 1 : 0, splits);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const int cx = pair ? 2 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cx, splits, 1);
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = attn_smem_bytes(d, pair);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cx;
  attr[0].val.clusterDim.y = splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void *fn = pair ? attn_kernel_fn<true>(d, paged) : attn_kernel_fn<false>(d, paged);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

AttnPlan plan_tree_attn(int B, int n_max, int Hq, int Hkv, int d, int64_t cap, int num_sms, bool paged,
                        int page_size) {
  AttnPlan pl{};
  const int g = Hq / Hkv;
  const int mt = (n_max * g + ATT_M - 1) / ATT_M;
  // Two or more M-tiles per (request, KV head) run as CTA pairs, which halve
  // the K/V bytes each SM receives per MMA (head_dim 128; paged caches with
  // pages of at most 64 tokens, so each CTA's 64 keys are whole pages).
  pl.pair = (d == 128 && mt >= 2 && (!paged || (page_size <= 64 && 64 % page_size == 0))) ? 1 : 0;
  if (pl.pair && max_active_clusters(d, paged, true, 1) < 1) pl.pair = 0;
  pl.mtiles = pl.pair ? 2 * ((mt + 1) / 2) : mt;
  pl.cap = cap;
  const int cx = pl.pair ? 2 : 1;
  const int max_splits = ATT_MAX_SPLITS / cx;
  const int64_t ctx_tiles = (cap + ATT_N - 1) / ATT_N;
  const int64_t tree_tiles = (n_max + ATT_N - 1) / ATT_N;
  const int64_t units = static_cast<int64_t>(B) * Hkv * (pl.mtiles / cx);   // clusters of one split
  const int64_t tot_tiles = ctx_tiles + tree_tiles;
  // KV splits per (b, kvh, M-tile or pair), up to a cluster of 16 CTAs
  // (non-portable sizes above 8 count only where the device keeps such
  // clusters resident): the count that minimises (waves of resident clusters)
  // x (tiles per CTA + a fixed cost of about four tiles for set-up, first
  // loads and the merge)
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= max_splits; ++s) {
    if (s > 1 && tot_tiles < 2LL * s) break;
    int per_wave = (s == 1 && !pl.pair) ? num_sms : max_active_clusters(d, paged, pl.pair != 0, s);
    if (per_wave < 1) continue;
    const int64_t waves = (units + per_wave - 1) / per_wave;
    const double cost = static_cast<double>(waves) * ((s > 1 ? 4.0 : 3.0) + (tot_tiles + s - 1) / s);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  // Paged caches: a 128-key tile arrives as 2 * (128 / page_size) small
  // copies per K or V, so a CTA streams its tiles several times slower than
  // from a contiguous cache, and the contexts of a paged batch are typically
  // ragged.  More, shorter splits (about four CTAs per SM over the batch)
  // balance the load better than the wave model above predicts: measured on a
  // 16-request batch of 512..8192-token contexts, 1 split 237 us, 2 splits
  // 199 us, 4 splits 187 us.
  if (paged) {
    const int64_t want = (4LL * num_sms / cx + units - 1) / units;
    int s_bal = static_cast<int>(std::min<int64_t>(max_splits, want));
    while (s_bal > best && tot_tiles < 2LL * s_bal) --s_bal;
    if (s_bal > best && max_active_clusters(d, paged, pl.pair != 0, s_bal) >= 1) best = s_bal;
  }
  pl.splits = best;
  pl.tiles_per_split = static_cast<int>((tot_tiles + best - 1) / best);
  if (pl.tiles_per_split == 0) pl.tiles_per_split = 1;
  // one partial slot per (b, kvh, M-tile, split) when the KV is split
  pl.ws_bytes = best > 1 ? static_cast<size_t>(B) * Hkv * pl.mtiles * best * (d / 4 + 1) * ATT_M * sizeof(float4) : 0;
  pl.off_o = pl.off_ml = 0;
  return pl;
}

cudaError_t prepare_tree_attn() {
  cudaError_t e;
  const void *fns[6] = {attn_kernel_fn<false>(128, false), attn_kernel_fn<false>(128, true),
                        attn_kernel_fn<false>(64, false),  attn_kernel_fn<false>(64, true),
                        attn_kernel_fn<true>(128, false),  attn_kernel_fn<true>(128, true)};
  const int smem[6] = {attn_smem_bytes(128, false), attn_smem_bytes(128, false), attn_smem_bytes(64, false),
                       attn_smem_bytes(64, false),  attn_smem_bytes(128, true),  attn_smem_bytes(128, true)};
  for (int i = 0; i < 6; ++i) {
    e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
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
                                float scale, bool paged, int page_size, int max_pages, int num_pages,
                                const int32_t *ctx_len, const int32_t *n, const uint64_t *mask,
                                const int32_t *block_table, void *out, void *ws, uint32_t *dev_err,
                                cudaStream_t stream) {
  AttnParams p{};
  p.part = reinterpret_cast<float4 *>(ws);
  p.B = B;
  p.n_max = n_max;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.mtiles = pl.mtiles;
  p.splits = pl.splits;
  p.tiles_per_split = pl.tiles_per_split;
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
  p.dev_err = dev_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.mtiles, pl.splits, B * Hkv);
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = attn_smem_bytes(d, pl.pair != 0);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  // the splits of one (b, kvh, M-tile) -- and the two CTAs of a pair -- form a cluster
  cfg.numAttrs = fill_launch_attrs(attr, pl.pair ? 2 : 1, pl.splits);
  if (pl.pair) {
    if (paged) return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<128, true, true>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
    return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<128, false, true>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
  }
  if (d == 128) {
    if (paged) return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<128, true, false>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
    return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<128, false, false>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
  }
  if (paged) return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<64, true, false>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<64, false, false>, maps[0], maps[1], maps[2], maps[3], maps[4], p);
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
