// Block pooling and per-request top-p block selection with sink/tail exemption.
//
// UniPrefill article, section 二 second step: average the token scores inside
// each block of G tokens, rank the blocks from most to least important and keep
// the smallest set whose importance sum reaches p of the total; exemption
// paragraph: blocks covering the first and last 128 tokens are always kept;
// section 三: the decision leaves the GPU as a binary mask.
//
// The selection itself (select_core.cuh) is deterministic: block masses are
// 48-bit fixed-point integers (relative to the request's largest block), the
// boundary score is found by an MSB-first radix select over the float bit
// patterns with integer histograms, and ties at the boundary score are taken
// in block-index order.
#include <cmath>

#include "select_core.cuh"
#include "upf_internal.cuh"

namespace upf {

namespace {

__device__ __forceinline__ int find_owner(const int32_t* off, int R, int x) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One warp per block: finalise token scores (sum of the per-group partials
// times 1/(H_q*n_eff)) or read given scores, then the block mean.
__global__ void __launch_bounds__(256) block_means_kernel(const SelectArgs a) {
  pdl_trigger();
  pdl_wait();
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  if (a.keep_bits) {
    const int nwords = (a.T + 31) / 32;
    for (int w = gtid; w < nwords; w += nthreads) a.keep_bits[w] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int nb_total = a.blk_off[a.R];
  for (int b = gtid >> 5; b < nb_total; b += nthreads >> 5) {
    const int r = find_owner(a.blk_off, a.R, b);
    const int i = b - a.blk_off[r];
    const int tok0 = a.cu[r];
    const int L = a.cu[r + 1] - tok0;
    const int lo = i * a.G, hi = min(L, lo + a.G);
    const float inv = 1.0f / float(a.Hq * min(a.n, L));
    float sum = 0.f;
    for (int t = lo + lane; t < hi; t += 32) {
      float v;
      if (a.P > 0) {
        v = 0.f;
        // partials in a fixed order; the unrolled loads are in flight together
#pragma unroll 8
        for (int c = 0; c < a.P; ++c) v += a.part[(int64_t)c * a.T + tok0 + t];
        v *= inv;
        if (a.scores_out) a.scores_out[tok0 + t] = v;
      } else {
        v = a.scores_in[tok0 + t];
      }
      sum += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) a.block_scores[b] = sum / float(hi - lo);
  }
}

// Per request: the shortest prefix of the blocks ranked by score (highest
// first, equal scores by lower index) whose running mass reaches top_p of the
// total (select_core.cuh), then the keep bits of its tokens: interior words by
// plain stores, the two words it may share with its neighbours by atomicOr
// (block_means_kernel cleared them).
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(const SelectArgs a, int nbp) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned char s_dyn[];
  const SelectScratch sc = carve_select(s_dyn, nbp);
  const int r = blockIdx.x, tid = threadIdx.x;
  const int b0 = a.blk_off[r];
  const int nb = a.blk_off[r + 1] - b0;
  const int tok0 = a.cu[r];
  const int L = a.cu[r + 1] - tok0;
  if (nb <= 0 || nb > nbp) {
    if (tid == 0) a.kept_count[r] = 0;
    return;
  }
  const int kept = select_request(a.block_scores + b0, nb, L, a.G, a.top_p, a.sink_keep, a.tail_keep, sc, a.status);
  const int w0 = tok0 >> 5, w1 = (tok0 + L - 1) >> 5;
  const int gshift = block_shift(a.G);
  for (int w = w0 + tid; w <= w1; w += blockDim.x) {
    const uint32_t bits = request_word_bits(sc.keep, tok0, L, a.G, gshift, w);
    const bool shared_word = (w * 32 < tok0) || (w * 32 + 32 > tok0 + L);
    if (shared_word) atomicOr(&a.keep_bits[w], bits);
    else a.keep_bits[w] = bits;
  }
  if (tid == 0) a.kept_count[r] = kept;
}


}  // namespace

cudaError_t launch_block_means(const SelectArgs& a, cudaStream_t s, bool pdl) {
  const int nwords = (a.T + 31) / 32;
  const int warps_needed = a.NB > 0 ? a.NB : 1;
  int blocks = (warps_needed + 7) / 8;
  blocks = max(blocks, (nwords + 255) / 256);
  blocks = min(max(blocks, 1), 4 * kPlanSMs * 8);
  return launch_kernel(block_means_kernel, blocks, 256, 0, s, pdl, a);
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s, bool pdl) {
  const int nbp = ((a.max_nb > 0 ? a.max_nb : 1) + 7) & ~7;
  const size_t smem = select_smem_bytes(nbp);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(select_kernel, a.R, kSelThreads, smem, s, pdl, a, nbp);
}

}  // namespace upf
