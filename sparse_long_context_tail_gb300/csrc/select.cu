// Block pooling and per-request top-p block selection with sink/tail exemption.
//
// UniPrefill article, section 二 second step: average the token scores inside
// each block of G tokens, rank the blocks from most to least important and keep
// the smallest set whose importance sum reaches p of the total; exemption
// paragraph: blocks covering the first and last 128 tokens are always kept;
// section 三: the decision leaves the GPU as a binary mask.
//
// Selection is deterministic: blocks are sorted by (score descending, index
// ascending) with a bitonic sort of 64-bit keys in shared memory, the running
// sums are float64 in a fixed association, and the boundary is the first sorted
// position whose running sum reaches top_p * (sum of all blocks).
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

// Orderable key: ascending order of the key = descending order of the float,
// ties broken by the lower block index.
__device__ __forceinline__ unsigned long long sort_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending-orderable
  u = ~u;                                           // descending
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(idx);
}

constexpr int kSelThreads = 1024;

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a, int n2) {
  extern __shared__ unsigned long long keys[];          // [n2]
  unsigned char* keep = reinterpret_cast<unsigned char*>(keys + n2);  // [n2]
  __shared__ double s_wsum[kSelThreads / 32];
  __shared__ int s_bad, s_k, s_cnt;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int b0 = a.blk_off[r];
  const int nb = a.blk_off[r + 1] - b0;
  const int tok0 = a.cu[r];
  const int L = a.cu[r + 1] - tok0;
  if (tid == 0) {
    s_bad = 0;
    s_k = nb;
    s_cnt = 0;
  }
  __syncthreads();
  if (nb <= 0 || nb > n2) {
    if (tid == 0) a.kept_count[r] = 0;
    return;
  }
  for (int i = tid; i < n2; i += blockDim.x) {
    if (i < nb) {
      const float v = a.block_scores[b0 + i];
      if (!isfinite(v)) s_bad = 1;
      keys[i] = sort_key(v, i);
    } else {
      keys[i] = ~0ull;
    }
    keep[i] = 0;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) set_status(a.status, UPF_ERR_NONFINITE);
    for (int i = tid; i < nb; i += blockDim.x) keep[i] = 1;
  } else {
    // Bitonic sort, ascending keys.
    for (int size = 2; size <= n2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < (n2 >> 1); i += blockDim.x) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const unsigned long long x = keys[lo], y = keys[hi];
          if ((x > y) == up) {
            keys[lo] = y;
            keys[hi] = x;
          }
        }
        __syncthreads();
      }
    }
    // Running sums in float64: thread t owns sorted positions [t*per, (t+1)*per).
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int p0 = min(nb, tid * per), p1 = min(nb, p0 + per);
    double local = 0.0;
    for (int p = p0; p < p1; ++p) local += double(a.block_scores[b0 + int(keys[p] & 0xffffffffu)]);
    // exclusive scan of `local` across the block (warp shuffles, then warp totals)
    const int lane = tid & 31, warp = tid >> 5;
    double incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      double w = lane < (int)(blockDim.x >> 5) ? s_wsum[lane] : 0.0;
      double wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < (int)(blockDim.x >> 5)) s_wsum[lane] = wi - w;  // exclusive warp offsets
    }
    __syncthreads();
    // The total is the running sum after all nb blocks, accumulated by the
    // owner of the last segment in exactly the order the search below uses, so
    // that with top_p = 1 the last running sum equals the target bit for bit.
    const int last_t = (nb - 1) / per;
    __shared__ double s_total;
    const double run0 = s_wsum[warp] + (incl - local);
    if (tid == last_t) {
      double t = run0;
      for (int p = p0; p < p1; ++p) t += double(a.block_scores[b0 + int(keys[p] & 0xffffffffu)]);
      s_total = t;
    }
    __syncthreads();
    const double target = double(a.top_p) * s_total;
    // smallest k >= 0 with cum_k >= target (cum_0 = 0)
    if (tid == 0 && 0.0 >= target) atomicMin(&s_k, 0);
    double run = run0;
    for (int p = p0; p < p1; ++p) {
      run += double(a.block_scores[b0 + int(keys[p] & 0xffffffffu)]);
      if (run >= target) {
        atomicMin(&s_k, p + 1);
        break;
      }
    }
    __syncthreads();
    const int k = s_k;
    for (int p = tid; p < k; p += blockDim.x) keep[int(keys[p] & 0xffffffffu)] = 1;
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
  atomicAdd(&s_cnt, cnt);
  // Keep bits of packed tokens [tok0, tok0 + L): interior words by plain
  // stores, the two words shared with neighbour requests by atomicOr.
  const int w0 = tok0 >> 5, w1 = (tok0 + L - 1) >> 5;
  for (int w = w0 + tid; w <= w1; w += blockDim.x) {
    uint32_t bits = 0;
    const int t_lo = max(tok0, w * 32), t_hi = min(tok0 + L, w * 32 + 32);
    for (int t = t_lo; t < t_hi; ++t)
      if (keep[(t - tok0) / a.G]) bits |= 1u << (t & 31);
    const bool shared_word = (w * 32 < tok0) || (w * 32 + 32 > tok0 + L);
    if (shared_word) atomicOr(&a.keep_bits[w], bits);
    else a.keep_bits[w] = bits;
  }
  __syncthreads();
  if (tid == 0) a.kept_count[r] = s_cnt;
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

cudaError_t launch_block_means(const SelectArgs& a, cudaStream_t s) {
  const int nwords = (a.T + 31) / 32;
  const int warps_needed = a.NB > 0 ? a.NB : 1;
  int blocks = (warps_needed + 7) / 8;
  blocks = max(blocks, (nwords + 255) / 256);
  blocks = min(max(blocks, 1), 4 * kPlanSMs * 8);
  block_means_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  const int n2 = next_pow2(a.max_nb > 0 ? a.max_nb : 1);
  const size_t smem = size_t(n2) * (sizeof(unsigned long long) + 1);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  select_kernel<<<a.R, kSelThreads, smem, s>>>(a, n2);
  return cudaGetLastError();
}

}  // namespace upf
