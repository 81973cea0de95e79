// Tensor-core (tcgen05 + TMEM + TMA) scoring passes for sm_103a.
//
// UniPrefill article, section 二 first step: the last n tokens act as
// questioners and score every token; section 三: scores and their online
// normalisation are computed on the GPU.  Both passes are dense bf16
// contractions of the group's tail queries with every key, so they run on the
// 5th-generation tensor cores with fp32 accumulators in TMEM:
//
//   pass 1 (queries as M): D[q, k] = Q_chunk[q, :] . K_tile[k, :]; every TMEM
//     lane is one query row, so the running max / sum of its causal softmax is
//     a per-thread reduction along the columns;
//   pass 2 (keys as M):    D[k, q] = K_tile[k, :] . Q_chunk[q, :]; every TMEM
//     lane is one key, so sum_q 2^(x*log2e*scale - lse2[q]) is a per-thread
//     reduction along the columns.
//
// One CTA per work item (request, kv head, query chunk, key split), 18 warps:
//   warps 0-15  epilogue (4 warpgroups; warp w reads TMEM lanes 32*(w%4)..)
//   warp 16     TMA producer (lane 0): the query chunk once, then the key
//               tiles, one 64-column slice (16 KB) per ring stage
//   warp 17     TMEM allocator + MMA issuer (lane 0)
// TMEM holds two 256-column slots; a "unit" (one key tile against one half of
// the query chunk) fills one slot while the epilogue drains the other.
// Every wait is bounded; on a timeout the kernel records UPF_ERR_TIMEOUT, the
// roles wind down, outstanding copies and MMAs are waited for (bounded), TMEM
// is freed and the kernel returns.
#include <cuda.h>

#include <cmath>

#include "sm100_ptx.cuh"
#include "upf_internal.cuh"

namespace upf {

namespace {

using namespace ptx;

constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;   // 512
constexpr int kThreadsTC = kEpiThreads + 64;  // + producer warp + MMA warp
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kTile = 128;                    // keys per tile
constexpr int kSliceBytes = kTile * 128;      // 128 rows x 64 bf16
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (about 2 s)

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
  it.s = local % nsplit;
  local /= nsplit;
  it.qc = local % NQC;
  it.g = local / NQC;
  return it;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

// Shared-memory plan of one CTA (same for both passes).
struct Smem {
  unsigned char* q;       // S slices x QCmax rows x 128 B
  unsigned char* stages;  // NS x 16 KB
  float* lse2;            // [QCmax]
  int* tq;                // [QCmax] query position in the request (pass 2)
  float* red;             // pass 2: [4 tiles][4 wg][128]; pass 1: float2 [4 wg][128]
  int* cnt;               // pass 2: [4 tiles][128] arrivals per key
  uint64_t* bars;         // full[NS], empty[NS], tfull[2], tempty[2], qfull, fin
  uint32_t* tmem_slot;
  int* abort_flag;
};

__host__ __device__ constexpr int stages_for(int d) { return d == 64 ? 8 : 5; }

__host__ __device__ inline size_t smem_bytes_tc(int d, int QCmax) {
  const int S = d / 64;
  const int NS = stages_for(d);
  size_t b = 1024;                                 // alignment slack
  b += size_t(S) * QCmax * 128;                    // Q chunk
  b += size_t(NS) * kSliceBytes;                   // K ring
  b += sizeof(float) * QCmax + sizeof(int) * QCmax;  // lse2, tq
  b += sizeof(float) * 4 * 4 * 128;                // red
  b += sizeof(int) * 4 * 128;                      // cnt
  b += sizeof(uint64_t) * (2 * NS + 6) + 16;       // barriers, tmem slot, abort flag
  return b;
}

__device__ __forceinline__ Smem carve(unsigned char* raw, int d, int QCmax) {
  Smem s;
  unsigned char* p = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int S = d / 64, NS = stages_for(d);
  s.q = p;
  p += size_t(S) * QCmax * 128;
  s.stages = p;
  p += size_t(NS) * kSliceBytes;
  s.lse2 = reinterpret_cast<float*>(p);
  p += sizeof(float) * QCmax;
  s.tq = reinterpret_cast<int*>(p);
  p += sizeof(int) * QCmax;
  s.red = reinterpret_cast<float*>(p);
  p += sizeof(float) * 4 * 4 * 128;
  s.cnt = reinterpret_cast<int*>(p);
  p += sizeof(int) * 4 * 128;
  s.bars = reinterpret_cast<uint64_t*>(p);
  p += sizeof(uint64_t) * (2 * NS + 6);
  s.tmem_slot = reinterpret_cast<uint32_t*>(p);
  s.abort_flag = reinterpret_cast<int*>(p + 8);
  return s;
}

// Rows of the query chunk present in this item: [0, rows_c); the MMA shapes
// use QCp = rows_c rounded up to 128 (zero rows beyond rows_c).
struct ChunkShape {
  int rows_c, QCp;
};

__device__ __forceinline__ ChunkShape chunk_shape(const ScoreArgs& a, int qc) {
  ChunkShape c;
  c.rows_c = min(a.QC, a.QR - qc * a.QC);
  c.QCp = ((c.rows_c + 127) / 128) * 128;
  return c;
}

// Producer: Q chunk (once), then key tiles slice by slice through the ring.
// Returns the number of key-slice loads issued.
__device__ int produce(const ScoreArgs& a, const CUtensorMap* tq_map, const CUtensorMap* tk_map, const Smem& sm,
                       const ItemTC& it, const ChunkShape& cs, int k0, int ntiles, int NS) {
  const int S = a.d / 64;
  const uint32_t qfull = smem_u32(&sm.bars[2 * NS + 4]);
  // Query rows: boxes of BQ rows of one head.
  const int BQ = a.q_box_rows;
  const int boxes = cs.rows_c / BQ;
  mbar_arrive_expect_tx(qfull, uint32_t(boxes) * S * BQ * 128);
  for (int b = 0; b < boxes; ++b) {
    const int rho = it.qc * a.QC + b * BQ;
    const int h = a.qhead[it.g * a.gamma + rho / a.n];
    const int tok = it.tok0 + it.L - a.n + rho % a.n;   // may be < 0 or in another request; masked later
    for (int s = 0; s < S; ++s)
      tma_load_3d(smem_u32(sm.q + size_t(s) * a.QC * 128 + size_t(b) * BQ * 128), tq_map, s * 64, h,
                  tok, qfull);
  }
  int iter = 0;
  for (int i = 0; i < ntiles; ++i) {
    for (int s = 0; s < S; ++s, ++iter) {
      const int st = iter % NS;
      const uint32_t ph = (iter / NS) & 1;
      if (*reinterpret_cast<volatile int*>(sm.abort_flag)) return iter;
      if (!mbar_wait(smem_u32(&sm.bars[NS + st]), ph ^ 1, kWaitLimit)) {
        set_status(a.status, UPF_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
        return iter;
      }
      const uint32_t full = smem_u32(&sm.bars[st]);
      mbar_arrive_expect_tx(full, kSliceBytes);
      tma_load_3d(smem_u32(sm.stages + size_t(st) * kSliceBytes), tk_map, s * 64, it.g, it.tok0 + k0 + i * kTile,
                  full);
    }
  }
  return iter;
}

// After an abort: wait (bounded) for the query load and for the last key
// load issued into each stage, so no copy is still landing when the CTA exits.
__device__ void drain_loads(const Smem& sm, int NS, int issued) {
  mbar_wait(smem_u32(&sm.bars[2 * NS + 4]), 0, kWaitLimit / 8);
  for (int st = 0; st < NS; ++st) {
    const int c = issued > st ? (issued - st + NS - 1) / NS : 0;   // loads issued into stage st
    if (c > 0) mbar_wait(smem_u32(&sm.bars[st]), (c - 1) & 1, kWaitLimit / 8);
  }
}

// ------------------------------------------------------------- pass 1 -----

__global__ void __launch_bounds__(kThreadsTC, 1)
    score_pass1_tc(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                   const __grid_constant__ ScoreArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x;
  if (item >= a.items1 || item >= a.item_off1[a.R]) return;
  const int d = a.d, S = d / 64, NS = stages_for(d);
  const Smem sm = carve(smem_raw, d, a.QC);
  const ItemTC it = locate_tc(a.item_off1, a.cu, a.R, item, a.KS1, a.NQC);
  const ChunkShape cs = chunk_shape(a, it.qc);
  const int k0 = it.s * a.KS1, k1 = min(it.L, k0 + a.KS1);
  const int ntiles = ceil_div_dev(k1 - k0, kTile);
  const int MT = cs.QCp / 128;            // M tiles of 128 query rows
  const int UM = MT >= 2 ? 2 : 1;         // M tiles per unit (one TMEM slot)
  const int H = (MT + 1) / 2;             // units per key tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&sm.bars[i]), 1);
      mbar_init(smem_u32(&sm.bars[NS + i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.bars[2 * NS + i]), 1);
      mbar_init(smem_u32(&sm.bars[2 * NS + 2 + i]), kEpiWarps);
    }
    mbar_init(smem_u32(&sm.bars[2 * NS + 4]), 1);
    mbar_init(smem_u32(&sm.bars[2 * NS + 5]), 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  // Zero the padding rows of the query chunk (generic stores, before any MMA reads them).
  for (int s = 0; s < S; ++s) {
    uint4* base = reinterpret_cast<uint4*>(sm.q + size_t(s) * a.QC * 128 + size_t(cs.rows_c) * 128);
    const int n16 = (cs.QCp - cs.rows_c) * 8;
    for (int i = tid; i < n16; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(sm.tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;

  int issued = 0;
  if (warp == kProducerWarp) {
    if (lane == 0) issued = produce(a, &tq_map, &tk_map, sm, it, cs, k0, ntiles, NS);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, kTile);
      bool ok = mbar_wait(smem_u32(&sm.bars[2 * NS + 4]), 0, kWaitLimit);
      int iter = 0, u = 0;
      for (int i = 0; ok && i < ntiles; ++i) {
        for (int s = 0; s < S && ok; ++s)
          ok = mbar_wait(smem_u32(&sm.bars[(iter + s) % NS]), ((iter + s) / NS) & 1, kWaitLimit);
        if (!ok) break;
        tc_fence_after();
        for (int h = 0; h < H && ok; ++h, ++u) {
          const int slot = u & 1;
          ok = mbar_wait(smem_u32(&sm.bars[2 * NS + 2 + slot]), ((u >> 1) & 1) ^ 1, kWaitLimit);
          if (!ok) break;
          tc_fence_after();
          for (int m = 0; m < UM && 2 * h + m < MT; ++m) {
            const uint32_t dt = tmem + uint32_t(slot * 256 + m * 128);
            for (int s = 0; s < S; ++s) {
              const uint32_t qa = smem_u32(sm.q + size_t(s) * a.QC * 128 + size_t(2 * h + m) * 128 * 128);
              const uint32_t kb = smem_u32(sm.stages + size_t((iter + s) % NS) * kSliceBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(dt, sdesc_kmajor_sw128(qa + kk * 32), sdesc_kmajor_sw128(kb + kk * 32), idesc,
                         (s | kk) ? 1u : 0u);
            }
          }
          mma_commit(smem_u32(&sm.bars[2 * NS + slot]));
        }
        for (int s = 0; s < S; ++s) mma_commit(smem_u32(&sm.bars[NS + (iter + s) % NS]));
        iter += S;
      }
      if (!ok) {
        set_status(a.status, UPF_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
      }
      // Wait for every MMA this thread issued before TMEM can be freed.
      mma_commit(smem_u32(&sm.bars[2 * NS + 5]));
      mbar_wait(smem_u32(&sm.bars[2 * NS + 5]), 0, kWaitLimit);
    }
  } else {
    // Epilogue: warpgroup wg, TMEM lane quadrant qd.
    const int wg = warp >> 2, qd = warp & 3;
    const int mrow = qd * 32 + lane;                 // row inside an M tile
    const int msel = UM == 2 ? (wg & 1) : 0;         // M tile inside the unit
    const int cw = UM == 2 ? 64 : 32;                // columns per warpgroup
    const int cbase = UM == 2 ? (wg >> 1) * 64 : wg * 32;
    float m_run[2] = {-INFINITY, -INFINITY}, z_run[2] = {0.f, 0.f};
    int t_row[2];
    for (int h = 0; h < 2; ++h) {
      const int row = (2 * h + msel) * 128 + mrow;   // row of the chunk
      const int rho = it.qc * a.QC + row;
      t_row[h] = (row < cs.rows_c) ? it.L - a.n + rho % a.n : -1;
    }
    const float sl = a.scale_log2;
    int u = 0;
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int kt = k0 + i * kTile;
      const bool masked_tile = kt + kTile - 1 > it.L - a.n;
      for (int h = 0; h < H; ++h, ++u) {
        const int slot = u & 1;
        if (*reinterpret_cast<volatile int*>(sm.abort_flag)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&sm.bars[2 * NS + slot]), (u >> 1) & 1, kWaitLimit)) {
          set_status(a.status, UPF_ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const bool have = 2 * h + msel < MT;
        float mloc = m_run[h], zloc = z_run[h];
        const int lim = t_row[h] - kt;               // columns c > lim are invisible
        for (int c0 = 0; c0 < cw; c0 += 32) {
          float v[32];
          tmem_ld32(tmem + (uint32_t(qd * 32) << 16) + uint32_t(slot * 256 + msel * 128 + cbase + c0), v);
          tmem_wait_ld();
          if (!have) continue;
          if (masked_tile) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cbase + c0 + j > lim) v[j] = -INFINITY;
          }
          float mx = v[0];
#pragma unroll
          for (int j = 1; j < 32; ++j) mx = fmaxf(mx, v[j]);
          if (mx == -INFINITY) continue;
          const float mxs = mx * sl;
          if (mxs > mloc) {
            zloc *= ex2_approx(mloc - mxs);
            mloc = mxs;
          }
          float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            z0 += ex2_approx(fmaf(v[j], sl, -mloc));
            z1 += ex2_approx(fmaf(v[j + 1], sl, -mloc));
            z2 += ex2_approx(fmaf(v[j + 2], sl, -mloc));
            z3 += ex2_approx(fmaf(v[j + 3], sl, -mloc));
          }
          zloc += (z0 + z1) + (z2 + z3);
        }
        m_run[h] = mloc;
        z_run[h] = zloc;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.bars[2 * NS + 2 + slot]));
      }
    }
    // Merge the (m, Z) of the warpgroups that covered the same rows, then store.
    float2* red = reinterpret_cast<float2*>(sm.red);   // [4 wg][128 rows] per half, reused per half
    for (int h = 0; h < 2; ++h) {
      epi_bar();
      red[wg * 128 + mrow] = make_float2(m_run[h], z_run[h]);
      epi_bar();
      const bool owner = UM == 2 ? (wg < 2) : (wg == 0);
      const int row = (2 * h + msel) * 128 + mrow;
      if (owner && 2 * h + msel < MT && row < cs.rows_c && (h == 0 || H == 2)) {
        float mm = -INFINITY;
        const int peers = UM == 2 ? 2 : 4;
        float2 p[4];
        for (int k = 0; k < peers; ++k) {
          p[k] = red[(UM == 2 ? (wg + 2 * k) : k) * 128 + mrow];
          mm = fmaxf(mm, p[k].x);
        }
        float zz = 0.f;
        if (mm > -INFINITY)
          for (int k = 0; k < peers; ++k)
            if (p[k].y > 0.f) zz += p[k].y * ex2_approx(p[k].x - mm);
        a.p1part[(int64_t)item * a.QC + row] = make_float2(mm, zz);
      }
    }
  }
  // Wind down: outstanding loads of an aborted pipeline, then free TMEM.
  if (warp == kProducerWarp && lane == 0 && *reinterpret_cast<volatile int*>(sm.abort_flag))
    drain_loads(sm, NS, issued);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------- pass 2 -----

__global__ void __launch_bounds__(kThreadsTC, 1)
    score_pass2_tc(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                   const __grid_constant__ ScoreArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x;
  if (item >= a.items2 || item >= a.item_off2[a.R]) return;
  const int d = a.d, S = d / 64, NS = stages_for(d);
  const Smem sm = carve(smem_raw, d, a.QC);
  const ItemTC it = locate_tc(a.item_off2, a.cu, a.R, item, a.KS2, a.NQC);
  const ChunkShape cs = chunk_shape(a, it.qc);
  const int k0 = it.s * a.KS2, k1 = min(it.L, k0 + a.KS2);
  const int ntiles = ceil_div_dev(k1 - k0, kTile);
  const int U = cs.QCp >= 256 ? 256 : cs.QCp;  // query columns per unit
  const int H = cs.QCp / U;                    // units per key tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&sm.bars[i]), 1);
      mbar_init(smem_u32(&sm.bars[NS + i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.bars[2 * NS + i]), 1);
      mbar_init(smem_u32(&sm.bars[2 * NS + 2 + i]), kEpiWarps);
    }
    mbar_init(smem_u32(&sm.bars[2 * NS + 4]), 1);
    mbar_init(smem_u32(&sm.bars[2 * NS + 5]), 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  for (int s = 0; s < S; ++s) {
    uint4* base = reinterpret_cast<uint4*>(sm.q + size_t(s) * a.QC * 128 + size_t(cs.rows_c) * 128);
    const int n16 = (cs.QCp - cs.rows_c) * 8;
    for (int i = tid; i < n16; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
  }
  for (int i = tid; i < 4 * 128; i += blockDim.x) sm.cnt[i] = 0;
  // lse2 of every query row of the chunk from the pass-1 partials; +inf marks
  // rows that do not exist (padding, or positions before the request start).
  if (tid < kEpiThreads) {
    const int nsplit1 = ceil_div_dev(it.L, a.KS1);
    const int64_t base1 = a.item_off1[it.r] + (int64_t)(it.g * a.NQC + it.qc) * nsplit1;
    for (int row = tid; row < cs.QCp; row += kEpiThreads) {
      float l2 = INFINITY;
      int t = -1;
      if (row < cs.rows_c) {
        const int rho = it.qc * a.QC + row;
        t = it.L - a.n + rho % a.n;
        float m = -INFINITY;
        for (int s = 0; s < nsplit1; ++s) m = fmaxf(m, a.p1part[(base1 + s) * a.QC + row].x);
        float Z = 0.f;
        if (m > -INFINITY)
          for (int s = 0; s < nsplit1; ++s) {
            const float2 p = a.p1part[(base1 + s) * a.QC + row];
            if (p.y > 0.f) Z += p.y * exp2f(p.x - m);
          }
        if (Z > 0.f && t >= 0) l2 = m + log2f(Z);
        else t = -1;
      }
      sm.lse2[row] = l2;
      sm.tq[row] = t;
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(sm.tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;

  int issued = 0;
  if (warp == kProducerWarp) {
    if (lane == 0) issued = produce(a, &tq_map, &tk_map, sm, it, cs, k0, ntiles, NS);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, U);
      bool ok = mbar_wait(smem_u32(&sm.bars[2 * NS + 4]), 0, kWaitLimit);
      int iter = 0, u = 0;
      for (int i = 0; ok && i < ntiles; ++i) {
        for (int s = 0; s < S && ok; ++s)
          ok = mbar_wait(smem_u32(&sm.bars[(iter + s) % NS]), ((iter + s) / NS) & 1, kWaitLimit);
        if (!ok) break;
        tc_fence_after();
        for (int h = 0; h < H && ok; ++h, ++u) {
          const int slot = u & 1;
          ok = mbar_wait(smem_u32(&sm.bars[2 * NS + 2 + slot]), ((u >> 1) & 1) ^ 1, kWaitLimit);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dt = tmem + uint32_t(slot * 256);
          for (int s = 0; s < S; ++s) {
            const uint32_t ka = smem_u32(sm.stages + size_t((iter + s) % NS) * kSliceBytes);
            const uint32_t qb = smem_u32(sm.q + size_t(s) * a.QC * 128 + size_t(h) * U * 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(dt, sdesc_kmajor_sw128(ka + kk * 32), sdesc_kmajor_sw128(qb + kk * 32), idesc,
                       (s | kk) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm.bars[2 * NS + slot]));
        }
        for (int s = 0; s < S; ++s) mma_commit(smem_u32(&sm.bars[NS + (iter + s) % NS]));
        iter += S;
      }
      if (!ok) {
        set_status(a.status, UPF_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
      }
      mma_commit(smem_u32(&sm.bars[2 * NS + 5]));
      mbar_wait(smem_u32(&sm.bars[2 * NS + 5]), 0, kWaitLimit);
    }
  } else {
    const int wg = warp >> 2, qd = warp & 3;
    const int krow = qd * 32 + lane;              // key inside the tile
    const int cw = U / 4;                         // columns per warpgroup per unit
    const float sl = a.scale_log2;
    float* out = a.part + (int64_t)(it.g * a.NQC + it.qc) * a.T + it.tok0;
    int u = 0;
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int kt = k0 + i * kTile;
      const int key = kt + krow;
      const bool masked_tile = kt + kTile - 1 > it.L - a.n;
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      for (int h = 0; h < H; ++h, ++u) {
        const int slot = u & 1;
        if (*reinterpret_cast<volatile int*>(sm.abort_flag)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&sm.bars[2 * NS + slot]), (u >> 1) & 1, kWaitLimit)) {
          set_status(a.status, UPF_ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const int cb = h * U + wg * cw;           // first chunk column of this warpgroup
        for (int c0 = 0; c0 < cw; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + (uint32_t(qd * 32) << 16) + uint32_t(slot * 256 + wg * cw + c0), v);
          tmem_wait_ld();
          const float4* l4 = reinterpret_cast<const float4*>(sm.lse2 + cb + c0);
          if (!masked_tile) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 l = l4[j / 4];
              acc0 += ex2_approx(fmaf(v[j], sl, -l.x));
              acc1 += ex2_approx(fmaf(v[j + 1], sl, -l.y));
              acc2 += ex2_approx(fmaf(v[j + 2], sl, -l.z));
              acc3 += ex2_approx(fmaf(v[j + 3], sl, -l.w));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = cb + c0 + j;
              if (key <= sm.tq[col]) acc0 += ex2_approx(fmaf(v[j], sl, -sm.lse2[col]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.bars[2 * NS + 2 + slot]));
      }
      if (!ok) break;
      // Combine the four warpgroups' column sums for this key without a
      // barrier: the last of the four to arrive adds them in a fixed order.
      volatile float* red = sm.red + (i & 3) * 512;
      int* cnt = sm.cnt + (i & 3) * 128;
      red[wg * 128 + krow] = (acc0 + acc1) + (acc2 + acc3);
      __threadfence_block();
      if (atomicAdd(&cnt[krow], 1) == 3) {
        __threadfence_block();
        const float tot = ((red[krow] + red[128 + krow]) + red[256 + krow]) + red[384 + krow];
        cnt[krow] = 0;
        if (key < k1) out[key] = tot;
      }
    }
  }
  if (warp == kProducerWarp && lane == 0 && *reinterpret_cast<volatile int*>(sm.abort_flag))
    drain_loads(sm, NS, issued);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
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

size_t score_tc_smem_bytes(int d, int QC) { return smem_bytes_tc(d, QC); }

cudaError_t launch_score_pass1_tc(const ScoreArgs& a, cudaStream_t s) {
  if (a.items1 == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.d, a.Hq, a.T, a.q_stride, a.q_box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.d, a.Hkv, a.T, a.k_stride, kTile)) != cudaSuccess) return e;
  const size_t smem = smem_bytes_tc(a.d, a.QC);
  if ((e = cudaFuncSetAttribute(score_pass1_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
    return e;
  score_pass1_tc<<<a.items1, kThreadsTC, smem, s>>>(mq, mk, a);
  return cudaGetLastError();
}

cudaError_t launch_score_pass2_tc(const ScoreArgs& a, cudaStream_t s) {
  if (a.items2 == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.d, a.Hq, a.T, a.q_stride, a.q_box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.d, a.Hkv, a.T, a.k_stride, kTile)) != cudaSuccess) return e;
  const size_t smem = smem_bytes_tc(a.d, a.QC);
  if ((e = cudaFuncSetAttribute(score_pass2_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
    return e;
  score_pass2_tc<<<a.items2, kThreadsTC, smem, s>>>(mq, mk, a);
  return cudaGetLastError();
}

}  // namespace upf
