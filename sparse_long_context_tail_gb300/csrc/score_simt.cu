// Batch descriptor kernel and the CUDA-core (fp32 FMA) scoring passes.
//
// UniPrefill article, section 二 first step (the last n tokens score every
// token) and section 三 (scores + online normalisation on the GPU).  Pass 1
// computes, per tail query, the running max and sum of its causal softmax over
// a key split; pass 2 merges those into the log-sum-exp, recomputes the logits
// and accumulates each key's normalised probability over the query rows of one
// kv group.  No logit matrix is stored.
#include <cmath>

#include "upf_internal.cuh"

namespace upf {

namespace {

__device__ __forceinline__ int ceil_div_dev(int a, int b) { return (a + b - 1) / b; }

// Largest r in [0, R) with off[r] <= x (off is non-decreasing, off[0] = 0).
__device__ __forceinline__ int find_owner(const int32_t* off, int R, int x) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct Item {
  int r, g, qc, s, tok0, L;
};

__device__ __forceinline__ Item locate(const int32_t* item_off, const int32_t* cu, int R, int item, int KS, int NQC) {
  Item it;
  it.r = find_owner(item_off, R, item);
  it.tok0 = cu[it.r];
  it.L = cu[it.r + 1] - it.tok0;
  const int nsplit = ceil_div_dev(it.L, KS);
  int local = item - item_off[it.r];
  it.s = local % nsplit;
  local /= nsplit;
  it.qc = local % NQC;
  it.g = local / NQC;
  return it;
}

// One warp: per-request item counts of both passes and block counts, scanned
// 32 requests at a time with shuffles.
__global__ void __launch_bounds__(32) describe_kernel(const DescribeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x;
  for (int i = lane; i < a.ncounters; i += 32) a.counters[i] = 0;
  bool bad = lane == 0 && (a.cu[0] != 0 || a.cu[a.R] != a.T);
  int carry[3] = {0, 0, 0};
  for (int base = 0; base < a.R; base += 32) {
    const int r = base + lane;
    int v[3] = {0, 0, 0};
    if (r < a.R) {
      const int L = a.cu[r + 1] - a.cu[r];
      bad |= L < 0;
      const int Lc = L < 0 ? 0 : L;
      v[0] = a.Hkv * a.NQC * ceil_div_dev(Lc, a.KS1);
      v[1] = a.Hkv * a.NQC2 * ceil_div_dev(Lc, a.KS2);
      v[2] = ceil_div_dev(Lc, a.G);
    }
    int incl[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        const int t = __shfl_up_sync(0xffffffffu, incl[c], o);
        if (lane >= o) incl[c] += t;
      }
    if (r < a.R) {
      a.item_off1[r] = carry[0] + incl[0] - v[0];
      a.item_off2[r] = carry[1] + incl[1] - v[1];
      a.blk_off[r] = carry[2] + incl[2] - v[2];
    }
#pragma unroll
    for (int c = 0; c < 3; ++c) carry[c] += __shfl_sync(0xffffffffu, incl[c], 31);
  }
  // The grids were sized on the host from cu_seqlens_host; a device copy that
  // disagrees must not drive any work.
  bad |= carry[0] != a.items1 || carry[1] != a.items2 || carry[2] != a.NB;
  bad = __any_sync(0xffffffffu, bad);
  if (bad) {
    for (int r = lane; r <= a.R; r += 32) a.item_off1[r] = a.item_off2[r] = a.blk_off[r] = 0;
    if (lane == 0) set_status(a.status, UPF_ERR_INVALID_ARG);
  } else if (lane == 0) {
    a.item_off1[a.R] = carry[0];
    a.item_off2[a.R] = carry[1];
    a.blk_off[a.R] = carry[2];
  }
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

constexpr int kThreads = 128;
constexpr int kKeyTile1 = 32;   // keys per shared-memory tile in pass 1
constexpr int kRowTile2 = 32;   // query rows per shared-memory tile in pass 2

// Pass 1: per item and query row, (m2, Z) of the causal softmax over the item's keys.
__global__ void __launch_bounds__(kThreads) score_pass1_simt(const __grid_constant__ ScoreArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float smem[];
  const int item = blockIdx.x;
  if (item >= a.item_off1[a.R] || item >= a.items1) return;
  const Item it = locate(a.item_off1, a.cu, a.R, item, a.KS1, a.NQC);
  const int d = a.d, tid = threadIdx.x;
  const int k0 = it.s * a.KS1, k1 = min(it.L, k0 + a.KS1);
  const int rows = min(a.QC, a.QR - it.qc * a.QC);
  float* qs = smem;                    // [kThreads][d+1]
  float* ks = smem + kThreads * (d + 1);  // [kKeyTile1][d]
  for (int sub = 0; sub < rows; sub += kThreads) {
    __syncthreads();
    for (int idx = tid; idx < kThreads * d; idx += kThreads) {
      const int rr = idx / d, e = idx % d;
      const int row = sub + rr;
      float v = 0.f;
      if (row < rows) {
        const int rho = it.qc * a.QC + row;
        const int h = a.qhead[it.g * a.gamma + rho / a.n];
        const int t = it.L - a.n + rho % a.n;
        if (t >= 0) v = bf2f(a.q[(int64_t)(it.tok0 + t) * a.q_stride + (int64_t)h * d + e]);
      }
      qs[rr * (d + 1) + e] = v;
    }
    const int row = sub + tid;
    const int rho = it.qc * a.QC + row;
    const int tq = it.L - a.n + rho % a.n;
    const bool valid = row < rows && tq >= 0;
    float m = -INFINITY, Z = 0.f;
    for (int kt = k0; kt < k1; kt += kKeyTile1) {
      __syncthreads();
      for (int idx = tid; idx < kKeyTile1 * d; idx += kThreads) {
        const int kk = idx / d, e = idx % d;
        const int key = kt + kk;
        ks[kk * d + e] = key < k1 ? bf2f(a.k[(int64_t)(it.tok0 + key) * a.k_stride + (int64_t)it.g * d + e]) : 0.f;
      }
      __syncthreads();
      float acc[kKeyTile1];
#pragma unroll
      for (int kk = 0; kk < kKeyTile1; ++kk) acc[kk] = 0.f;
      for (int e = 0; e < d; ++e) {
        const float qv = qs[tid * (d + 1) + e];
#pragma unroll
        for (int kk = 0; kk < kKeyTile1; ++kk) acc[kk] = fmaf(qv, ks[kk * d + e], acc[kk]);
      }
#pragma unroll
      for (int kk = 0; kk < kKeyTile1; ++kk) {
        const int key = kt + kk;
        if (valid && key < k1 && key <= tq) {
          const float x = acc[kk] * a.scale_log2;
          if (x > m) {
            Z = Z * exp2f(m - x) + 1.f;
            m = x;
          } else {
            Z += exp2f(x - m);
          }
        }
      }
    }
    if (row < rows) a.p1part[(int64_t)item * a.QC + row] = make_float2(m, Z);
  }
}

// Pass 2: per key, sum over the rows of one query chunk of 2^(x - lse2).
__global__ void __launch_bounds__(kThreads) score_pass2_simt(const __grid_constant__ ScoreArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float smem[];
  const int item = blockIdx.x;
  if (item >= a.item_off2[a.R] || item >= a.items2) return;
  const Item it = locate(a.item_off2, a.cu, a.R, item, a.KS2, a.NQC);
  const int d = a.d, tid = threadIdx.x;
  const int k0 = it.s * a.KS2, k1 = min(it.L, k0 + a.KS2);
  const int rows = min(a.QC, a.QR - it.qc * a.QC);
  float* lse = smem;                          // [QC]
  float* ks = lse + a.QC;                     // [kThreads][d+1]
  float* qs = ks + kThreads * (d + 1);        // [kRowTile2][d]
  // Merge the pass-1 partials of (r, g, qc) into lse2 per row.
  const int nsplit1 = ceil_div_dev(it.L, a.KS1);
  const int64_t base1 = a.item_off1[it.r] + (int64_t)(it.g * a.NQC + it.qc) * nsplit1;
  for (int row = tid; row < rows; row += kThreads) {
    float m = -INFINITY;
    for (int s = 0; s < nsplit1; ++s) m = fmaxf(m, a.p1part[(base1 + s) * a.QC + row].x);
    float Z = 0.f;
    if (m > -INFINITY)
      for (int s = 0; s < nsplit1; ++s) {
        const float2 p = a.p1part[(base1 + s) * a.QC + row];
        if (p.y > 0.f) Z += p.y * exp2f(p.x - m);
      }
    lse[row] = Z > 0.f ? m + log2f(Z) : INFINITY;
  }
  for (int kt = k0; kt < k1; kt += kThreads) {
    __syncthreads();
    for (int idx = tid; idx < kThreads * d; idx += kThreads) {
      const int kk = idx / d, e = idx % d;
      const int key = kt + kk;
      ks[kk * (d + 1) + e] =
          key < k1 ? bf2f(a.k[(int64_t)(it.tok0 + key) * a.k_stride + (int64_t)it.g * d + e]) : 0.f;
    }
    const int key = kt + tid;
    float acc_key = 0.f;
    for (int rb = 0; rb < rows; rb += kRowTile2) {
      __syncthreads();
      for (int idx = tid; idx < kRowTile2 * d; idx += kThreads) {
        const int rr = idx / d, e = idx % d;
        const int row = rb + rr;
        float v = 0.f;
        if (row < rows) {
          const int rho = it.qc * a.QC + row;
          const int h = a.qhead[it.g * a.gamma + rho / a.n];
          const int t = it.L - a.n + rho % a.n;
          if (t >= 0) v = bf2f(a.q[(int64_t)(it.tok0 + t) * a.q_stride + (int64_t)h * d + e]);
        }
        qs[rr * d + e] = v;
      }
      __syncthreads();
      float dot[kRowTile2];
#pragma unroll
      for (int rr = 0; rr < kRowTile2; ++rr) dot[rr] = 0.f;
      for (int e = 0; e < d; ++e) {
        const float kv = ks[tid * (d + 1) + e];
#pragma unroll
        for (int rr = 0; rr < kRowTile2; ++rr) dot[rr] = fmaf(kv, qs[rr * d + e], dot[rr]);
      }
#pragma unroll
      for (int rr = 0; rr < kRowTile2; ++rr) {
        const int row = rb + rr;
        if (row < rows) {
          const int rho = it.qc * a.QC + row;
          const int tq = it.L - a.n + rho % a.n;
          if (key < k1 && key <= tq) acc_key += exp2f(dot[rr] * a.scale_log2 - lse[row]);
        }
      }
    }
    if (key < k1) a.part[(int64_t)(it.g * a.NQC + it.qc) * a.T + it.tok0 + key] = acc_key;
  }
}

size_t pass1_smem(int d) { return sizeof(float) * (kThreads * (d + 1) + kKeyTile1 * d); }
size_t pass2_smem(int d, int QC) { return sizeof(float) * (QC + kThreads * (d + 1) + kRowTile2 * d); }

}  // namespace

cudaError_t launch_describe(const DescribeArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(describe_kernel, 1, 32, 0, s, pdl, a);
}

cudaError_t launch_score_pass1(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  if (a.use_tc) return a.use_pair ? launch_score_pass1_pair(a, s, pdl) : launch_score_pass1_tc(a, s, pdl);
  if (a.items1 == 0) return cudaSuccess;
  const size_t smem = pass1_smem(a.d);
  cudaError_t e = cudaFuncSetAttribute(score_pass1_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(score_pass1_simt, a.items1, kThreads, smem, s, pdl, a);
}

cudaError_t launch_score_pass2(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  if (a.use_tc) return a.use_pair ? launch_score_pass2_pair(a, s, pdl) : launch_score_pass2_tc(a, s, pdl);
  if (a.items2 == 0) return cudaSuccess;
  const size_t smem = pass2_smem(a.d, a.QC);
  cudaError_t e = cudaFuncSetAttribute(score_pass2_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(score_pass2_simt, a.items2, kThreads, smem, s, pdl, a);
}

}  // namespace upf
