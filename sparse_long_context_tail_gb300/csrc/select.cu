// Block pooling and per-request top-p block selection with sink/tail exemption.
//
// UniPrefill article, section 二 second step: average the token scores inside
// each block of G tokens, rank the blocks from most to least important and keep
// the smallest set whose importance sum reaches p of the total; exemption
// paragraph: blocks covering the first and last 128 tokens are always kept;
// section 三: the decision leaves the GPU as a binary mask.
//
// Selection is deterministic: block masses are 48-bit fixed-point integers
// (relative to the request's largest block), the boundary score is found by an
// MSB-first radix select over the float bit patterns with integer histograms,
// and ties at the boundary score are taken in block-index order.  The rounding
// of the masses is below 1e-10 of the total.
#include <cmath>

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

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

// 2^e as a float, for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Block masses as 48-bit fixed point relative to the largest block of the
// request: m = floor(v * 2^(48 - ex)) with vmax = f * 2^ex, f in [0.5, 1), so
// every m < 2^48 and a request's total (<= 16384 blocks) stays below 2^62.
// The scaling is by powers of two only (two steps keep each factor normal).
__device__ __forceinline__ unsigned long long fixed_mass(float v, int sh) {
  const int s1 = min(sh, 127);
  return __float2ull_rz((v * pow2f(s1)) * pow2f(sh - s1));
}

template <typename T>
__device__ __forceinline__ T block_reduce_sum(T v, T* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s_tmp[warp] = v;
  __syncthreads();
  T t = 0;
  for (int w = 0; w < kSelWarps; ++w) t += s_tmp[w];   // fixed order
  __syncthreads();
  return t;
}

// Per request: the shortest prefix of the blocks ranked by score (highest
// first, equal scores by lower index) whose running mass reaches top_p of the
// total, found without sorting.  Non-negative float bit patterns order like
// the values, so an MSB-first radix select over the 32-bit patterns (8 bits per
// round) finds the score v* of the last block needed; blocks above v* are in,
// and blocks equal to v* are taken in index order until the mass is reached.
// All masses are integers, so every sum is exact and independent of order.
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a, int nbp) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned long long s_m[];                       // [nbp] fixed-point masses
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_m + nbp);       // [nbp] float bits
  unsigned char* keep = reinterpret_cast<unsigned char*>(s_bits + nbp);  // [nbp]
  __shared__ unsigned long long h_mass[256];
  __shared__ unsigned int h_cnt[256];
  __shared__ unsigned long long s_u64[kSelWarps];
  __shared__ float s_f[kSelWarps];
  __shared__ int s_i[kSelWarps];
  __shared__ int s_digit, s_cnt;
  __shared__ unsigned long long s_above;
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b0 = a.blk_off[r];
  const int nb = a.blk_off[r + 1] - b0;
  const int tok0 = a.cu[r];
  const int L = a.cu[r + 1] - tok0;
  if (nb <= 0 || nb > nbp) {
    if (tid == 0) a.kept_count[r] = 0;
    return;
  }
  // Load, validate (finite and >= 0) and find the largest score.
  float vmax = 0.f;
  int bad = 0;
  for (int i = tid; i < nb; i += blockDim.x) {
    const float v = a.block_scores[b0 + i];
    bad |= !(isfinite(v) && v >= 0.f);
    s_bits[i] = __float_as_uint(v);
    vmax = fmaxf(vmax, v);
    keep[i] = 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    s_f[warp] = vmax;
    s_i[warp] = bad;
  }
  __syncthreads();
  vmax = 0.f;
  bad = 0;
  for (int w = 0; w < kSelWarps; ++w) {
    vmax = fmaxf(vmax, s_f[w]);
    bad |= s_i[w];
  }
  if (tid == 0) s_cnt = 0;
  if (bad) {
    if (tid == 0) set_status(a.status, UPF_ERR_NONFINITE);
    for (int i = tid; i < nb; i += blockDim.x) keep[i] = 1;
  } else {
    int ex = 0;
    if (vmax > 0.f) frexpf(vmax, &ex);
    const int sh = 48 - ex;
    unsigned long long part = 0;
    for (int i = tid; i < nb; i += blockDim.x) {
      const unsigned long long m = vmax > 0.f ? fixed_mass(__uint_as_float(s_bits[i]), sh) : 0ull;
      s_m[i] = m;
      part += m;
    }
    const unsigned long long total = block_reduce_sum(part, s_u64);
    // Mass the selected prefix must reach: the smallest integer >= top_p * total.
    const unsigned long long target = (unsigned long long)ceil((double)a.top_p * (double)total);
    if (target > 0) {
      uint32_t prefix = 0, pmask = 0;
      unsigned long long above = 0;   // mass of blocks ranked strictly before the candidates
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int d = tid; d < 256; d += blockDim.x) {
          h_mass[d] = 0;
          h_cnt[d] = 0;
        }
        __syncthreads();
        for (int i = tid; i < nb; i += blockDim.x) {
          const uint32_t bits = s_bits[i];
          if ((bits & pmask) == prefix) {
            const int d = (bits >> shift) & 255;
            atomicAdd(&h_mass[d], s_m[i]);
            atomicAdd(&h_cnt[d], 1u);
          }
        }
        __syncthreads();
        if (warp == 0) {
          // Buckets from the highest digit down; lane l owns digits 255-8l .. 248-8l.
          unsigned long long loc[8], lsum = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            loc[j] = h_mass[255 - 8 * lane - j];
            lsum += loc[j];
          }
          unsigned long long incl = lsum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          const unsigned long long base = above + incl - lsum;   // mass before this lane's digits
          const bool hit = base + lsum >= target && base < target;
          const unsigned int who = __ballot_sync(0xffffffffu, hit);
          const int src = who ? __ffs(who) - 1 : 31;
          if (lane == src) {
            unsigned long long run = base;
            int dsel = 255 - 8 * lane - 7;
            for (int j = 0; j < 8; ++j) {
              if (run + loc[j] >= target) {
                dsel = 255 - 8 * lane - j;
                break;
              }
              run += loc[j];
            }
            s_digit = dsel;
            s_above = run;
          }
        }
        __syncthreads();
        prefix |= uint32_t(s_digit) << shift;
        pmask |= 255u << shift;
        above = s_above;
        __syncthreads();
      }
      // prefix = bits of the boundary score v*.  Blocks above it are in; the
      // tied ones (equal scores) enter in index order until the mass suffices.
      // Thread t owns the contiguous index range [t*per, (t+1)*per).
      const int per = (nb + blockDim.x - 1) / blockDim.x;
      const int i0 = min(nb, tid * per), i1 = min(nb, i0 + per);
      int ties = 0;
      unsigned long long w = 0;
      for (int i = i0; i < i1; ++i) {
        const uint32_t bits = s_bits[i];
        if (bits > prefix) keep[i] = 1;
        else if (bits == prefix) {
          ++ties;
          w = s_m[i];
        }
      }
      // exclusive scan of tie counts in index order
      int incl = ties;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) s_i[warp] = incl;
      __syncthreads();
      int before = incl - ties;
      for (int ww = 0; ww < warp; ++ww) before += s_i[ww];
      if (ties > 0) {
        // every tied block carries the same mass w > 0 (the boundary bucket reached the target)
        const unsigned long long need = target - above;
        const unsigned long long take = w > 0 ? (need + w - 1) / w : 0;
        int rank = before;
        for (int i = i0; i < i1; ++i)
          if (s_bits[i] == prefix) {
            if ((unsigned long long)rank < take) keep[i] = 1;
            ++rank;
          }
      }
    }
  }
  __syncthreads();
  // Exempt blocks: overlap with [0, sink) or [L - tail, L).
  const int sink_hi = min(a.sink_keep, L);
  const int tail_lo = max(0, L - a.tail_keep);
  for (int i = tid; i < nb; i += blockDim.x) {
    const int lo = i * a.G, hi = min(L, lo + a.G);
    if (lo < sink_hi || hi > tail_lo) keep[i] = 1;
  }
  __syncthreads();
  // Kept tokens.
  int cnt = 0;
  for (int i = tid; i < nb; i += blockDim.x)
    if (keep[i]) cnt += min(L, (i + 1) * a.G) - i * a.G;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0 && cnt) atomicAdd(&s_cnt, cnt);
  // Keep bits of packed tokens [tok0, tok0 + L): interior words by plain
  // stores, the two words shared with neighbour requests by atomicOr.
  const int w0 = tok0 >> 5, w1 = (tok0 + L - 1) >> 5;
  for (int w = w0 + tid; w <= w1; w += blockDim.x) {
    uint32_t bits = 0;
    const int t_lo = max(tok0, w * 32), t_hi = min(tok0 + L, w * 32 + 32);
    // walk the blocks that overlap this word's tokens
    for (int t = t_lo; t < t_hi;) {
      const int blk = (t - tok0) / a.G;
      const int t_end = min(t_hi, tok0 + (blk + 1) * a.G);
      if (keep[blk]) {
        const int len = t_end - t;
        bits |= (len >= 32 ? 0xffffffffu : ((1u << len) - 1u)) << (t & 31);
      }
      t = t_end;
    }
    const bool shared_word = (w * 32 < tok0) || (w * 32 + 32 > tok0 + L);
    if (shared_word) atomicOr(&a.keep_bits[w], bits);
    else a.keep_bits[w] = bits;
  }
  __syncthreads();
  if (tid == 0) a.kept_count[r] = s_cnt;
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
  const size_t smem = size_t(nbp) * (sizeof(unsigned long long) + sizeof(uint32_t) + 1);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(select_kernel, a.R, kSelThreads, smem, s, pdl, a, nbp);
}

}  // namespace upf
