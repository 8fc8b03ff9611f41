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
// split).  The M rows pack g = Hq/Hkv query heads x tree nodes of one KV head
// (GQA), so every K/V tile is used by all heads of its group.  Roles:
//   warp 4      TMA producer: Q once, then K/V tiles (128 keys) into a 2-stage
//               ring with 128-byte swizzle; paged caches are gathered page by
//               page through a 4-D tensor map; no multicast.
//   warp 5      MMA issuer (one thread): S = Q K^T into TMEM (two S buffers),
//               O += P V with P read from TMEM (P aliases its S buffer).
//   warps 0-3   softmax: thread r owns TMEM lane r = M-tile row r; it reads S,
//               applies the context bound or the ancestor bits, keeps the
//               running max / sum in the log2 domain, writes P (bf16) to TMEM,
//               rescales O when the max grows, and runs the epilogue.
// Splits of the context combine in the workspace: the last CTA of a
// (b, kvh, M-tile) (atomic ticket, no waiting) merges the partial (O, m, l).
// Every mbarrier wait is bounded in time; on expiry the CTA records
// BASTION_DEVERR_TIMEOUT, drains what it issued and frees its TMEM.
//
// f32 path: an exact fp32 flash-decoding kernel, one CTA per (b, node, head).
#include <math_constants.h>

#include <algorithm>

#include "sm100_ptx.cuh"

namespace bst {

constexpr int ATT_THREADS = 192;
constexpr int ATT_N = 128;            // keys per tile
constexpr int ATT_M = 128;            // rows per M-tile
constexpr int ATT_HALF = ATT_N * 128; // bytes of 128 rows x 64 bf16
constexpr uint64_t ATT_WAIT_NS = 200ull * 1000ull * 1000ull;

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
  float *ws_o;               // [units, splits, 128, d]
  float2 *ws_ml;             // [units, splits, 128]
  uint32_t *tickets;         // [units]
  uint32_t *dev_err;
};

struct AttnBars {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last;
};

template <int D>
struct AttnLayout {
  static constexpr int NH = D / 64;
  static constexpr int Q_BYTES = NH * ATT_HALF;
  static constexpr int KV_BYTES = NH * ATT_HALF;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int Q_OFF = 0;
  static constexpr int STAGE_OFF = Q_BYTES;
  static constexpr int BAR_OFF = STAGE_OFF + 2 * STAGE_BYTES;
  static constexpr int USED = BAR_OFF + static_cast<int>(sizeof(AttnBars));
  // 1024 bytes of slack for aligning the dynamic shared memory base; at least
  // 120 KB so that a single CTA owns each SM (its TMEM allocation is 512 columns).
  static constexpr int SMEM = (USED + 1024) > 120 * 1024 ? (USED + 1024) : 120 * 1024;
};

// Optional phase trace (compiled in with -DBST_TRACE only): %globaltimer
// stamps at the pipeline's phase boundaries, 32 per CTA, read back with
// bastion_trace_read().  Normal builds contain none of it.
#ifdef BST_TRACE
__device__ unsigned long long g_attn_trace[4096 * 32];
#define BST_TRACE_AT(ev)                                                                                  \
  do {                                                                                                  \
    const unsigned cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);               \
    if (cta_ < 4096u && (ev) < 32) g_attn_trace[cta_ * 32u + (ev)] = globaltimer_ns();                 \
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

template <int D, bool kPaged>
__global__ void __launch_bounds__(ATT_THREADS, 1) tree_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kt,
    const __grid_constant__ CUtensorMap tm_vt, const AttnParams p) {
  using LY = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + LY::Q_OFF;
  AttnBars *bars = reinterpret_cast<AttnBars *>(smem + LY::BAR_OFF);
  volatile int *abort = &bars->abort;

  const int mtile = blockIdx.x;
  const int split = blockIdx.y;
  const int bh = blockIdx.z;
  const int b = bh / p.Hkv;
  const int kvh = bh - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int unit = bh * p.mtiles + mtile;

  if (tid == 0) BST_TRACE_AT(0);
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

  const int ctx_tiles = (L + ATT_N - 1) / ATT_N;
  const int ct0 = split * p.tiles_per_split;
  const int n_ctx = max(0, min(ctx_tiles, ct0 + p.tiles_per_split) - ct0);
  const int n_tree = (split == 0) ? (nb + ATT_N - 1) / ATT_N : 0;
  const int T = n_ctx + n_tree;

  // row owned by a softmax thread
  const int r = tid;   // valid for tid < 128
  const int pidx = mtile * ATT_M + r;
  const int node = pidx / p.g;
  const int hl = pidx - node * p.g;
  const bool active = (tid < 128) && (node < nb);

  float m_run = -CUDART_INF_F;
  float l_run = 0.f;
  bool ok = true;

  if (T > 0) {
    if (tid == 0) {
      mbar_init(&bars->q_full, 1);
      mbar_init(&bars->kv_full[0], 1);
      mbar_init(&bars->kv_full[1], 1);
      mbar_init(&bars->kv_empty[0], 1);
      mbar_init(&bars->kv_empty[1], 1);
      mbar_init(&bars->s_full[0], 1);
      mbar_init(&bars->s_full[1], 1);
      mbar_init(&bars->p_full[0], 128);
      mbar_init(&bars->p_full[1], 128);
      mbar_init(&bars->o_done, 1);
      mbar_init(&bars->drain, 1);
      bars->abort = 0;
      bars->last = 0;
      fence_mbar_init();
    }
    if (warp == 0) {
      tmem_alloc(&bars->tmem_base, 512);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    const uint32_t tO = tbase + 256;
    if (tid == 0) BST_TRACE_AT(1);

    if (warp == 4) {
      // ------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_kt);
        tma_prefetch_desc(&tm_vt);
        BST_TRACE_AT(2);
        mbar_expect_tx(&bars->q_full, LY::Q_BYTES);
#pragma unroll
        for (int h = 0; h < LY::NH; ++h)
          tma_load_3d(sQ + h * ATT_HALF, &tm_q, &bars->q_full, h * 64, kvh * p.g, b * p.n_max + mtile * (ATT_M / p.g));
        int issued = 0;
        for (int j = 0; j < T; ++j) {
          const int st = j & 1;
          if (j >= 2 && !mbar_wait(&bars->kv_empty[st], ((j >> 1) - 1) & 1, abort, ATT_WAIT_NS)) break;
          uint8_t *sK = smem + LY::STAGE_OFF + st * LY::STAGE_BYTES;
          uint8_t *sV = sK + LY::KV_BYTES;
          uint64_t *fb = &bars->kv_full[st];
          mbar_expect_tx(fb, LY::STAGE_BYTES);
          if (j < n_ctx) {
            const int ct = ct0 + j;
            if (!kPaged) {
#pragma unroll
              for (int h = 0; h < LY::NH; ++h) {
                tma_load_3d(sK + h * ATT_HALF, &tm_k, fb, h * 64, ct * ATT_N, b * p.Hkv + kvh);
                tma_load_3d(sV + h * ATT_HALF, &tm_v, fb, h * 64, ct * ATT_N, b * p.Hkv + kvh);
              }
            } else {
              const int ps = p.page_size;
              for (int pi = 0; pi < ATT_N / ps; ++pi) {
                const int tok = ct * ATT_N + pi * ps;
                int page = p.num_pages;   // out of range: the copy reads zeros
                if (tok < L) {
                  page = p.block_table[static_cast<int64_t>(b) * p.max_pages + tok / ps];
                  if (page < 0 || page >= p.num_pages) {
                    set_err(p.dev_err, BASTION_DEVERR_PAGE);
                    page = p.num_pages;
                  }
                }
#pragma unroll
                for (int h = 0; h < LY::NH; ++h) {
                  tma_load_4d(sK + h * ATT_HALF + pi * ps * 128, &tm_k, fb, h * 64, 0, kvh, page);
                  tma_load_4d(sV + h * ATT_HALF + pi * ps * 128, &tm_v, fb, h * 64, 0, kvh, page);
                }
              }
            }
          } else {
            const int tt = j - n_ctx;
#pragma unroll
            for (int h = 0; h < LY::NH; ++h) {
              tma_load_3d(sK + h * ATT_HALF, &tm_kt, fb, h * 64, kvh, b * p.n_max + tt * ATT_N);
              tma_load_3d(sV + h * ATT_HALF, &tm_vt, fb, h * 64, kvh, b * p.n_max + tt * ATT_N);
            }
          }
          issued = j + 1;
        }
        if (*abort) {
          // let the copies already in flight land before the CTA goes away
          for (int j = max(0, issued - 2); j < issued; ++j)
            mbar_wait(&bars->kv_full[j & 1], (j >> 1) & 1, abort, ATT_WAIT_NS);
          mbar_wait(&bars->q_full, 0, abort, ATT_WAIT_NS);
        }
      }
    } else if (warp == 5) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t IDESC_QK = idesc_bf16(ATT_M, ATT_N, 0);
        constexpr uint32_t IDESC_PV = idesc_bf16(ATT_M, D, 1);
        const uint32_t q_addr = smem_u32(sQ);
        bool any = false;
        auto issue_pv = [&](int jj) -> bool {
          const int sb = jj & 1;
          if (!mbar_wait(&bars->p_full[sb], (jj >> 1) & 1, abort, ATT_WAIT_NS)) return false;
          tc_fence_after();
          const uint32_t v_addr = smem_u32(smem + LY::STAGE_OFF + sb * LY::STAGE_BYTES + LY::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < ATT_N / 16; ++kk) {
            // V is the MN-major B operand: 8 keys per 1024-byte swizzle group,
            // the two 64-column halves of d are ATT_HALF bytes apart.
            const uint64_t bdesc = sdesc_sw128(v_addr + kk * 2048, ATT_HALF, 1024);
            mma_ts(tO, tbase + sb * 128 + kk * 8, bdesc, IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->o_done);
          mma_commit(&bars->kv_empty[sb]);
          return true;
        };
        bool run = mbar_wait(&bars->q_full, 0, abort, ATT_WAIT_NS);
        tc_fence_after();
        for (int j = 0; run && j < T; ++j) {
          const int st = j & 1;
          if (!mbar_wait(&bars->kv_full[st], (j >> 1) & 1, abort, ATT_WAIT_NS)) { run = false; break; }
          if (j >= 2 && !mbar_wait(&bars->o_done, (j - 2) & 1, abort, ATT_WAIT_NS)) { run = false; break; }
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + LY::STAGE_OFF + st * LY::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int h = kk >> 2;
            const uint32_t off = h * ATT_HALF + (kk & 3) * 32;
            const uint64_t adesc = sdesc_sw128(q_addr + off, 16, 1024);
            const uint64_t bdesc = sdesc_sw128(k_addr + off, 16, 1024);
            mma_ss(tbase + st * 128, adesc, bdesc, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          any = true;
          mma_commit(&bars->s_full[st]);
          BST_TRACE_AT(3 + min(j, 7));
          if (j >= 1 && !issue_pv(j - 1)) { run = false; break; }
        }
        if (run) issue_pv(T - 1);
        if (any) {
          // every MMA issued above has finished before TMEM is released
          mma_commit(&bars->drain);
          mbar_wait(&bars->drain, 0, abort, ATT_WAIT_NS);
        }
      }
    } else {
      // ------------------------------------------------ softmax warps 0-3
      const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
      const int W = (p.n_max + 63) >> 6;
      unsigned long long mw[4] = {0ull, 0ull, 0ull, 0ull};
      if (active) {
        const unsigned long long *mrow = p.mask + (static_cast<int64_t>(b) * p.n_max + node) * W;
        for (int w = 0; w < W; ++w) mw[w] = mrow[w];
      }
      for (int j = 0; j < T; ++j) {
        const int sb = j & 1;
        if (!warp_wait(&bars->s_full[sb], (j >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        if (tid == 0) BST_TRACE_AT(11 + min(j, 7));
        uint32_t s[ATT_N];
        tmem_ld32(tbase + lane_off + sb * 128 + 0, s + 0);
        tmem_ld32(tbase + lane_off + sb * 128 + 32, s + 32);
        tmem_ld32(tbase + lane_off + sb * 128 + 64, s + 64);
        tmem_ld32(tbase + lane_off + sb * 128 + 96, s + 96);
        tmem_wait_ld32(s + 0);
        tmem_wait_ld32(s + 32);
        tmem_wait_ld32(s + 64);
        tmem_wait_ld32(s + 96);
        // masking: context tiles bound by L, tree tiles by the ancestor bits;
        // the scaled, masked scores overwrite s in place
        float tmax = -CUDART_INF_F;
        if (j < n_ctx) {
          const int nvalid = L - (ct0 + j) * ATT_N;
#pragma unroll
          for (int c = 0; c < ATT_N; ++c) {
            const float v = (c < nvalid) ? __uint_as_float(s[c]) * p.scale_log2 : -CUDART_INF_F;
            s[c] = __float_as_uint(v);
            tmax = fmaxf(tmax, v);
          }
        } else {
          const int tt = j - n_ctx;
          const unsigned long long w0 = (tt == 0) ? mw[0] : mw[2];
          const unsigned long long w1 = (tt == 0) ? mw[1] : mw[3];
#pragma unroll
          for (int c = 0; c < ATT_N; ++c) {
            const unsigned long long w = (c < 64) ? w0 : w1;
            const bool vis = ((w >> (c & 63)) & 1ull) != 0ull;
            const float v = vis ? __uint_as_float(s[c]) * p.scale_log2 : -CUDART_INF_F;
            s[c] = __float_as_uint(v);
            tmax = fmaxf(tmax, v);
          }
        }
        const float m_new = fmaxf(m_run, tmax);
        const float msub = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        const float alpha = exp2f(m_run - msub);
        float sum = 0.f;
        uint32_t pk[ATT_N / 2];
#pragma unroll
        for (int c = 0; c < ATT_N; c += 2) {
          const float p0 = exp2f(__uint_as_float(s[c]) - msub);
          const float p1 = exp2f(__uint_as_float(s[c + 1]) - msub);
          sum += p0 + p1;
          pk[c >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tbase + lane_off + sb * 128 + 0, pk + 0);
        tmem_st32(tbase + lane_off + sb * 128 + 32, pk + 32);
        l_run = l_run * alpha + sum;
        const bool need = (j >= 1) && (alpha != 1.f);
        if (__any_sync(FULL, need)) {
          // O must hold P_{j-1} V_{j-1} before it is rescaled
          if (!warp_wait(&bars->o_done, (j - 1) & 1, abort)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + cc * 32, o);
            tmem_wait_ld32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + lane_off + cc * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
        if (tid == 0) BST_TRACE_AT(19 + min(j, 7));
        m_run = m_new;
      }
      // ---- epilogue: O after the last P V
      float o[D];
      // the drain barrier completes once, after the last P V (and every MMA
      // before it) has finished
      if (ok && !warp_wait(&bars->drain, 0, abort)) ok = false;
      if (tid == 0) BST_TRACE_AT(27);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t t32[32];
          tmem_ld32(tO + lane_off + cc * 32, t32);
          tmem_wait_ld32(t32);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[cc * 32 + e] = __uint_as_float(t32[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < D; ++e) o[e] = 0.f;
      }
      if (p.splits == 1) {
        if (ok && active) {
          const float inv = 1.f / l_run;
          uint16_t *dst = p.out + ((static_cast<int64_t>(b) * p.n_max + node) * p.Hq + kvh * p.g + hl) * D;
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            uint4 v;
            v.x = pack_bf16x2(o[c + 0] * inv, o[c + 1] * inv);
            v.y = pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
            v.z = pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
            v.w = pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
            *reinterpret_cast<uint4 *>(dst + c) = v;
          }
        }
      } else {
        const int64_t prow = (static_cast<int64_t>(unit) * p.splits + split) * ATT_M + r;
        float *dst = p.ws_o + prow * D;
#pragma unroll
        for (int c = 0; c < D; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
        p.ws_ml[prow] = make_float2(ok ? m_run : -CUDART_INF_F, ok ? l_run : 0.f);
        if (tid == 0) BST_TRACE_AT(28);
      }
    }
    // all roles done with TMEM
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, 512);
    if (tid == 0) BST_TRACE_AT(31);
    if (*abort && tid == 0) set_err(p.dev_err, BASTION_DEVERR_TIMEOUT);
  } else if (p.splits > 1 && tid < 128) {
    // nothing to attend to in this split: an empty partial
    const int64_t prow = (static_cast<int64_t>(unit) * p.splits + split) * ATT_M + r;
    p.ws_ml[prow] = make_float2(-CUDART_INF_F, 0.f);
  }

  // ---- split combine: the last CTA of this (b, kvh, M-tile) merges
  if (p.splits > 1) {
    __shared__ int s_last;
    if (tid < 128) {
      __threadfence();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (tid == 0) s_last = (atomicAdd(&p.tickets[unit], 1u) == static_cast<uint32_t>(p.splits - 1)) ? 1 : 0;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (s_last) {
        __threadfence();
        if (tid == 0) BST_TRACE_AT(29);
        if (active) {
          const int64_t base = static_cast<int64_t>(unit) * p.splits * ATT_M + r;
          float M = -CUDART_INF_F;
          for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(&p.ws_ml[base + s * ATT_M].x));
          float acc[D];
#pragma unroll
          for (int e = 0; e < D; ++e) acc[e] = 0.f;
          float lsum = 0.f;
          for (int s = 0; s < p.splits; ++s) {
            const float2 ml = __ldcg(&p.ws_ml[base + s * ATT_M]);
            if (ml.x == -CUDART_INF_F) continue;
            const float w = exp2f(ml.x - M);
            lsum += w * ml.y;
            const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + (base + s * ATT_M) * D);
#pragma unroll
            for (int c = 0; c < D / 4; ++c) {
              const float4 v = __ldcg(src + c);
              acc[4 * c + 0] += w * v.x;
              acc[4 * c + 1] += w * v.y;
              acc[4 * c + 2] += w * v.z;
              acc[4 * c + 3] += w * v.w;
            }
          }
          const float inv = 1.f / lsum;
          uint16_t *dst = p.out + ((static_cast<int64_t>(b) * p.n_max + node) * p.Hq + kvh * p.g + hl) * D;
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            uint4 v;
            v.x = pack_bf16x2(acc[c + 0] * inv, acc[c + 1] * inv);
            v.y = pack_bf16x2(acc[c + 2] * inv, acc[c + 3] * inv);
            v.z = pack_bf16x2(acc[c + 4] * inv, acc[c + 5] * inv);
            v.w = pack_bf16x2(acc[c + 6] * inv, acc[c + 7] * inv);
            *reinterpret_cast<uint4 *>(dst + c) = v;
          }
        }
        if (tid == 0) p.tickets[unit] = 0u;   // ready for the next call
        if (tid == 0) BST_TRACE_AT(30);
      }
    }
  }
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

__global__ void __launch_bounds__(128) tree_attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ kt,
                                                            const float *__restrict__ vt, const float *__restrict__ kc,
                                                            const float *__restrict__ vc, float *__restrict__ out,
                                                            const AttnParamsF32 p) {
  const int h = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
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
  __shared__ float qs[128];
  __shared__ float ps[128];
  __shared__ float red[4];
  if (tid < p.d) qs[tid] = q[((static_cast<int64_t>(b) * p.n_max + i) * p.Hq + h) * p.d + tid];
  __syncthreads();
  float m = -CUDART_INF_F, l = 0.f, acc = 0.f;
  const int total = L + nb;
  for (int base = 0; base < total; base += 128) {
    const int j = base + tid;
    float s = -CUDART_INF_F;
    if (j < L) {
      bool okp = true;
      const float *kr = f32_ctx_row(kc, p, b, kvh, j, &okp);
      if (okp) {
        float a = 0.f;
        for (int e = 0; e < p.d; ++e) a = fmaf(qs[e], kr[e], a);
        s = a * p.scale;
      } else {
        set_err(p.dev_err, BASTION_DEVERR_PAGE);
      }
    } else if (j < total) {
      const int jt = j - L;
      if ((mrow[jt >> 6] >> (jt & 63)) & 1ull) {
        const float *kr = kt + ((static_cast<int64_t>(b) * p.n_max + jt) * p.Hkv + kvh) * p.d;
        float a = 0.f;
        for (int e = 0; e < p.d; ++e) a = fmaf(qs[e], kr[e], a);
        s = a * p.scale;
      }
    }
    float cm = warp_max_f(s);
    if ((tid & 31) == 0) red[tid >> 5] = cm;
    __syncthreads();
    cm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const float m_new = fmaxf(m, cm);
    if (m_new == -CUDART_INF_F) continue;   // uniform: nothing visible yet
    const float alpha = expf(m - m_new);
    const float pj = (s == -CUDART_INF_F) ? 0.f : expf(s - m_new);
    ps[tid] = pj;
    float cs = warp_sum_f(pj);
    if ((tid & 31) == 0) red[tid >> 5] = cs;
    __syncthreads();
    cs = red[0] + red[1] + red[2] + red[3];
    l = l * alpha + cs;
    acc *= alpha;
    const int cnt = min(128, total - base);
    if (tid < p.d) {
      for (int jj = 0; jj < cnt; ++jj) {
        const float w = ps[jj];
        if (w == 0.f) continue;
        const int jk = base + jj;
        const float *vr;
        if (jk < L) {
          bool okp = true;
          vr = f32_ctx_row(vc, p, b, kvh, jk, &okp);
          if (!okp) continue;
        } else {
          vr = vt + ((static_cast<int64_t>(b) * p.n_max + (jk - L)) * p.Hkv + kvh) * p.d;
        }
        acc = fmaf(w, vr[tid], acc);
      }
    }
    m = m_new;
    __syncthreads();
  }
  if (tid < p.d) out[((static_cast<int64_t>(b) * p.n_max + i) * p.Hq + h) * p.d + tid] = acc / l;
}

// ------------------------------------------------------------------ host side
struct AttnPlan {
  int mtiles, splits, tiles_per_split;
  int64_t cap;
  size_t ws_bytes, off_o, off_ml;
};

AttnPlan plan_tree_attn(int B, int n_max, int Hq, int Hkv, int d, int64_t cap, int num_sms) {
  AttnPlan pl{};
  const int g = Hq / Hkv;
  pl.mtiles = (n_max * g + ATT_M - 1) / ATT_M;
  pl.cap = cap;
  const int64_t ctx_tiles = (cap + ATT_N - 1) / ATT_N;
  const int64_t units = static_cast<int64_t>(B) * Hkv * pl.mtiles;
  // enough CTAs to fill the GPU about twice, at least 4 tiles per split
  int64_t splits = (2LL * num_sms + units - 1) / units;
  splits = std::min<int64_t>(splits, std::max<int64_t>(1, ctx_tiles / 4));
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, 64));
  pl.splits = static_cast<int>(splits);
  pl.tiles_per_split = static_cast<int>((ctx_tiles + splits - 1) / splits);
  if (pl.tiles_per_split == 0) pl.tiles_per_split = 1;
  if (pl.splits == 1) {
    pl.ws_bytes = 0;
  } else {
    const size_t t = (static_cast<size_t>(units) * 4 + 255) / 256 * 256;
    pl.off_o = t;
    pl.off_ml = t + static_cast<size_t>(units) * pl.splits * ATT_M * d * 4;
    pl.ws_bytes = pl.off_ml + static_cast<size_t>(units) * pl.splits * ATT_M * 8;
  }
  return pl;
}

cudaError_t prepare_tree_attn() {
  cudaError_t e;
  e = cudaFuncSetAttribute(tree_attn_tc_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnLayout<128>::SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tree_attn_tc_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnLayout<128>::SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tree_attn_tc_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnLayout<64>::SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tree_attn_tc_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnLayout<64>::SMEM);
}

cudaError_t launch_tree_attn_tc(const CUtensorMap *maps, const AttnPlan &pl, int B, int n_max, int Hq, int Hkv, int d,
                                float scale, bool paged, int page_size, int max_pages, int num_pages,
                                const int32_t *ctx_len, const int32_t *n, const uint64_t *mask,
                                const int32_t *block_table, void *out, void *ws, uint32_t *dev_err,
                                cudaStream_t stream) {
  AttnParams p{};
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
  if (pl.splits > 1) {
    p.tickets = reinterpret_cast<uint32_t *>(ws);
    p.ws_o = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + pl.off_o);
    p.ws_ml = reinterpret_cast<float2 *>(reinterpret_cast<char *>(ws) + pl.off_ml);
  }
  p.dev_err = dev_err;
  dim3 grid(pl.mtiles, pl.splits, B * Hkv);
  if (d == 128) {
    if (paged)
      tree_attn_tc_kernel<128, true><<<grid, ATT_THREADS, AttnLayout<128>::SMEM, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
    else
      tree_attn_tc_kernel<128, false><<<grid, ATT_THREADS, AttnLayout<128>::SMEM, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  } else {
    if (paged)
      tree_attn_tc_kernel<64, true><<<grid, ATT_THREADS, AttnLayout<64>::SMEM, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
    else
      tree_attn_tc_kernel<64, false><<<grid, ATT_THREADS, AttnLayout<64>::SMEM, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  }
  return cudaGetLastError();
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
  tree_attn_f32_kernel<<<dim3(Hq, n_max, B), 128, 0, stream>>>(q, kt, vt, kc, vc, out, p);
  return cudaGetLastError();
}

}  // namespace bst
