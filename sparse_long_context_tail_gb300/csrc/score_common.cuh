// Pieces shared by the tensor-core scoring kernels (one CTA per work item in
// score_tc.cu, a CTA pair per work item in score_pair.cu): work-item
// location, the epilogue's exponential sums, and the TMA descriptors.
//
// UniPrefill article, section 二 first step (the last n tokens score every
// token) and section 三 (scores and their online normalisation on the GPU).
#pragma once

#include <cuda.h>

#include <climits>
#include <cmath>

#include "sm100_ptx.cuh"
#include "upf_internal.cuh"

namespace upf {

namespace {

using namespace ptx;

__host__ __device__ constexpr int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int imax(int a, int b) { return a > b ? a : b; }
__device__ __forceinline__ int ceil_div_dev(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int find_owner(const int32_t* off, int R, int x) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Work item: request r, kv head g, key split s, query chunk qc.  Items of one
// request are numbered ((g * nsplit) + s) * NQC + qc, so the chunks that share
// a key range are neighbours in the grid and read the range once from DRAM.
struct ItemTC {
  int r, g, qc, s, tok0, L;
};

__device__ __forceinline__ ItemTC locate_tc(const int32_t* item_off, const int32_t* cu, int R, int item, int KS,
                                            int NQC) {
  ItemTC it;
  it.r = find_owner(item_off, R, item);
  it.tok0 = cu[it.r];
  it.L = cu[it.r + 1] - it.tok0;
  const int nsplit = ceil_div_dev(it.L, KS);
  int local = item - item_off[it.r];
  it.qc = local % NQC;
  local /= NQC;
  it.s = local % nsplit;
  it.g = local / nsplit;
  return it;
}

__device__ __forceinline__ int64_t item_index(const int32_t* item_off, int r, int g, int s, int qc, int nsplit,
                                              int NQC) {
  return item_off[r] + ((int64_t)g * nsplit + s) * NQC + qc;
}

// Work item `item` of pass 1 (pass2 false) or pass 2 and the first pass-1
// item of a row group, from the tables carried in the parameters (a must be
// the kernel's __grid_constant__ parameter) or else the workspace tables
// describe_kernel wrote.  Each branch reads its own tables directly: a pointer
// chosen at run time between the two spaces costs the epilogue warps
// registers they do not have (measured: spills in both passes).
__device__ __forceinline__ bool item_exists(const ScoreArgs& a, int item, bool pass2) {
  if (item >= (pass2 ? a.items2 : a.items1)) return false;
  if (a.desc.R > 0) return item < (pass2 ? a.desc.off2[a.R] : a.desc.off1[a.R]);
  return item < (pass2 ? a.item_off2[a.R] : a.item_off1[a.R]);
}
__device__ __forceinline__ ItemTC locate_item(const ScoreArgs& a, int item, bool pass2) {
  if (a.desc.R > 0) return locate_tc(pass2 ? a.desc.off2 : a.desc.off1, a.desc.cu, a.R, item, pass2 ? a.KS2 : a.KS1, a.NQC);
  return locate_tc(pass2 ? a.item_off2 : a.item_off1, a.cu, a.R, item, pass2 ? a.KS2 : a.KS1, a.NQC);
}
__device__ __forceinline__ int64_t pass1_item_index(const ScoreArgs& a, int r, int g, int qc, int nsplit1) {
  if (a.desc.R > 0) return item_index(a.desc.off1, r, g, 0, qc, nsplit1, a.NQC1);
  return item_index(a.item_off1, r, g, 0, qc, nsplit1, a.NQC1);
}

// Pass 2's entry for chunk row `row` of item it: -lse2 of the row's query,
// merged from the pass-1 partials (m2, Z) of all nsplit1 key splits, and the
// query's position; -inf and -1 for rows that do not exist (padding, or
// positions before the request start).  Up to 24 partials are loaded before
// any is used (a load feeding each step would expose one L2 latency per
// split), the largest m2 is taken first, then the rescaled sums are added;
// ex2.approx and lg2.approx move the result by about 1e-7 relative.
// The part of a row's merge that reads only the parameters (and tables
// written before pass 1): the address of its first partial and its query
// position (t = -1: no row).  Pass 2 does it before waiting for pass 1.
struct LseRow {
  const float2* src;
  int t;
};

__device__ __forceinline__ LseRow lse_row_prep(const ScoreArgs& a, const ItemTC& it, int row, int rows_c, int nsplit1) {
  LseRow p{nullptr, -1};
  if (row < rows_c) {
    const int gr = it.qc * a.QC + row;   // row of the group; pass 1 may cut the group into smaller chunks
    const int qc1 = a.QC1 == a.QC ? it.qc : gr / a.QC1;
    p.t = it.L - a.n + gr % a.n;
    p.src = a.p1part + pass1_item_index(a, it.r, it.g, qc1, nsplit1) * a.QC1 + (gr - qc1 * a.QC1);
  }
  return p;
}

// The merge itself (split_stride: consecutive splits of one (g, qc)).
__device__ __forceinline__ void lse_row_finish(const LseRow& p, int nsplit1, int64_t split_stride, float& nlse,
                                               int& tq) {
  float l2 = INFINITY;
  int t = p.t;
  if (p.src) {
    const float2* src = p.src;
    float mm = -INFINITY, Z = 0.f;
    for (int s0 = 0; s0 < nsplit1; s0 += 24) {
      float2 pp[24];
#pragma unroll
      for (int k = 0; k < 24; ++k)
        pp[k] = s0 + k < nsplit1 ? src[(s0 + k) * split_stride] : make_float2(-INFINITY, 0.f);
      float mb = -INFINITY;
#pragma unroll
      for (int k = 0; k < 24; ++k)
        if (pp[k].y > 0.f) mb = fmaxf(mb, pp[k].x);
      if (mb > mm) {
        Z = mm > -INFINITY ? Z * ex2_approx(mm - mb) : 0.f;
        mm = mb;
      }
#pragma unroll
      for (int k = 0; k < 24; ++k)
        if (pp[k].y > 0.f) Z += pp[k].y * ex2_approx(pp[k].x - mm);
    }
    if (Z > 0.f && t >= 0) l2 = mm + lg2_approx(Z);
    else t = -1;
  }
  nlse = -l2;
  tq = t;
}

__device__ __forceinline__ void chunk_row_lse(const ScoreArgs& a, const ItemTC& it, int row, int rows_c, int nsplit1,
                                              float& nlse, int& tq) {
  lse_row_finish(lse_row_prep(a, it, row, rows_c, nsplit1), nsplit1, (int64_t)a.NQC1 * a.QC1, nlse, tq);
}

// With carried tables, one warp of pass 1's first CTA does what
// describe_kernel does otherwise: it checks the device cu_seqlens against the
// host's (a disagreement is reported; every kernel addresses the batch through
// the carried tables, so it cannot move any work out of bounds) and clears
// the tail kernel's counters, which run only after pass 2 has finished.
__device__ __forceinline__ void desc_check(const ScoreArgs& a, int lane) {
  if (a.desc.R <= 0) return;
  bool bad = false;
  for (int i = lane; i <= a.desc.R; i += 32) bad |= a.cu[i] != a.desc.cu[i];
  for (int i = lane; i < a.ncounters; i += 32) a.counters[i] = 0;
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(a.status, UPF_ERR_INVALID_ARG);
}

// ------------------------------------------------------- epilogue math -----

// sum_j 2^(v[j] * sl - ref) over 32 values, with the affine step and the
// accumulation in packed fp32 pairs.
__device__ __forceinline__ float exp_sum32(const float (&v)[32], float sl, float ref) {
  const uint64_t sl2 = pack2(sl, sl), nm2 = pack2(-ref, -ref);
  uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    float a, b, c, d;
    unpack2(fma2(pack2(v[j], v[j + 1]), sl2, nm2), a, b);
    unpack2(fma2(pack2(v[j + 2], v[j + 3]), sl2, nm2), c, d);
    acc0 = add2(acc0, pack2(ex2_approx(a), ex2_approx(b)));
    acc1 = add2(acc1, pack2(ex2_approx(c), ex2_approx(d)));
  }
  float lo, hi;
  unpack2(add2(acc0, acc1), lo, hi);
  return lo + hi;
}

__device__ __forceinline__ float max32(const float (&v)[32]) {
  float t[11];
#pragma unroll
  for (int j = 0; j < 10; ++j) t[j] = max3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
  t[10] = fmaxf(v[30], v[31]);
  return fmaxf(max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), max3(t[6], t[7], t[8])), fmaxf(t[9], t[10]));
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(addr));
  return r;
}

// Pass 1 folds the logits of one query row (raw dot products; invisible
// entries -inf) into its running (m, Z), m and the exponents in log2 units
// scaled by sl = scale * log2(e), Z = sum 2^(x*sl - m).  m is a reference
// point, not the running maximum: the exponentials are taken against the
// current m, and only a unit whose chunk sums leave [0, 2^20] (a term above
// about 2^15, an overflow, or the first visible chunk, where m is -inf and a
// sum is inf or NaN) takes this slow step, which moves m to the maximum of the
// unit's CPW chunks (if above m) and rescales Z.  m + log2 Z is the same
// either way.
template <int CPW>
__device__ __forceinline__ void online_rescale(const float (&va)[32], const float (&vb)[32], float sl, float& m,
                                               float& z) {
  const float mx = (CPW == 2 ? fmaxf(max32(va), max32(vb)) : max32(va)) * sl;
  if (mx == -INFINITY) return;        // nothing visible
  const float mn = fmaxf(m, mx);
  float sum = exp_sum32(va, sl, mn);
  if (CPW == 2) sum += exp_sum32(vb, sl, mn);
  z = z * ex2_approx(m - mn) + sum;
  m = mn;
}

// Pass-2 step, unmasked: acc += 2^(v * sl - lse2) over 32 query columns of one
// key; nlse is the shared-memory address of -lse2 of those columns (16-byte
// aligned).
__device__ __forceinline__ void normalised_sum32(const float (&v)[32], uint32_t nlse, float sl, uint64_t& acc0,
                                                 uint64_t& acc1) {
  const uint64_t sl2 = pack2(sl, sl);
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 l = lds_f4(nlse + 4 * j);
    float a, b, c, d;
    unpack2(fma2(pack2(v[j], v[j + 1]), sl2, pack2(l.x, l.y)), a, b);
    unpack2(fma2(pack2(v[j + 2], v[j + 3]), sl2, pack2(l.z, l.w)), c, d);
    acc0 = add2(acc0, pack2(ex2_approx(a), ex2_approx(b)));
    acc1 = add2(acc1, pack2(ex2_approx(c), ex2_approx(d)));
  }
}

// The same near the causal edge: only the columns whose query sees the key.
__device__ __forceinline__ float normalised_sum32_masked(const float (&v)[32], const float* nlse, const int* tq,
                                                         int key, float sl) {
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (key <= tq[j]) acc += ex2_approx(fmaf(v[j], sl, nlse[j]));
  return acc;
}

// ------------------------------------------------------------- host -------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D bf16 map over [T, H, d] rows (row stride `stride` elements): box of 64
// dims x 1 head x `rows` tokens, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, int d, int H, int T, int64_t stride, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(H), cuuint64_t(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(stride) * 2};
  cuuint32_t box[3] = {64, 1, cuuint32_t(rows)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

}  // namespace upf
