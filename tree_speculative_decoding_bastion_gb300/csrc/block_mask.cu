// Block-diffusion drafter mask.
//
// FlexDraft page ("FlexDraft: Flexible Speculative Decoding via Attention
// Tuning and Bonus-Guided Calibration"), "Attention-Tuning": mask tokens are
// appended to the clean prefix; in the deep layers they attend bidirectionally
// inside their block and to the clean prefix, and stay isolated from other
// blocks.  BASTION ("Bastion: Budget-Aware Speculative Decoding with
// Tree-structured Block Diffusion Drafting"), Methodik §1: one drafter pass
// fills a block of positions.
//
// The attention itself is bastion_tree_attn with the clean prefix as the
// context and the block positions as the "tree" rows; this kernel writes the
// mask it takes: for request b and row i < n[b], bit j of mask[b, i, :] is set
// iff j < n[b] and i / block == j / block.  Rows i >= n[b] are zero.
//
// Design: one thread per 64-bit mask word; a word's bits are the
// intersection of [64 w, 64 w + 64) with the row's block [lo, hi), written as
// a shifted run of ones.  Pure integer work, a few KB per call.
#include "common.cuh"

namespace bst {

constexpr int BM_THREADS = 256;

__global__ void __launch_bounds__(BM_THREADS) block_mask_kernel(int n_max, int W, int block,
                                                                const int32_t *__restrict__ n,
                                                                unsigned long long *__restrict__ mask,
                                                                uint32_t *__restrict__ dev_err) {
  const int b = blockIdx.y;
  pdl_wait();   // n may come from the previous stage
  int nb = n[b];
  if (nb < 1 || nb > n_max) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_err(dev_err, BASTION_DEVERR_N);
    nb = 0;   // every row of the request is cleared
  }
  pdl_trigger();
  const int words = n_max * W;
  for (int t = blockIdx.x * BM_THREADS + threadIdx.x; t < words; t += gridDim.x * BM_THREADS) {
    const int i = t / W;
    const int w = t % W;
    unsigned long long bits = 0ull;
    if (i < nb) {
      const int lo = max(i / block * block, 64 * w);
      const int hi = min(min(nb, (i / block + 1) * block), 64 * w + 64);
      if (hi > lo) {
        const int len = hi - lo;   // 1..64
        const unsigned long long run = len == 64 ? ~0ull : ((1ull << len) - 1ull);
        bits = run << (lo - 64 * w);
      }
    }
    mask[static_cast<int64_t>(b) * words + t] = bits;
  }
}

cudaError_t launch_block_mask(int B, int n_max, int block, const int32_t *n, uint64_t *mask, uint32_t *dev_err,
                              cudaStream_t stream) {
  const int W = (n_max + 63) / 64;
  const int words = n_max * W;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((words + BM_THREADS - 1) / BM_THREADS, B, 1);
  cfg.blockDim = dim3(BM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = fill_launch_attrs(attr);
  return cudaLaunchKernelEx(&cfg, block_mask_kernel, n_max, W, block, n,
                            reinterpret_cast<unsigned long long *>(mask), dev_err);
}

}  // namespace bst
