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
// A "unit" is one 128-key tile against one group of 128 query rows (pass 1)
// or columns (pass 2): a 128 x 128 fp32 accumulator, one of four TMEM slots.
// Warpgroup pair P (warpgroups 2P, 2P+1) owns every other group and drains
// slots P and P+2 in turn, so the MMA fills a pair's next slot while the pair
// reduces the current one, and the two pairs run out of phase.
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

constexpr int kSlots = 4;      // TMEM slots of 128 fp32 columns
constexpr int kRedTiles = 8;   // pass-2 key tiles whose warpgroup sums may be in flight

// Shared-memory plan of one CTA (same for both passes).
struct Smem {
  unsigned char* q;       // S slices x QCmax rows x 128 B
  unsigned char* stages;  // NS x 16 KB
  float* lse2;            // [QCmax] (pass 2: -lse2)
  int* tq;                // [QCmax] query position in the request (pass 2)
  float* red;             // pass 2: [kRedTiles][4 wg][128]; pass 1: float2 [4 wg][2][128]
  int* cnt;               // pass 2: [kRedTiles][128] arrivals per key
  uint64_t* bars;         // full[NS], empty[NS], tfull[4], tempty[4], qfull, fin
  uint32_t* tmem_slot;
  int* abort_flag;
};

__host__ __device__ constexpr int stages_for(int d) { return d == 64 ? 8 : 4; }

__host__ __device__ inline size_t smem_bytes_tc(int d, int QCmax) {
  const int S = d / 64;
  const int NS = stages_for(d);
  size_t b = 1024;                                     // alignment slack
  b += size_t(S) * QCmax * 128;                        // Q chunk
  b += size_t(NS) * kSliceBytes;                       // K ring
  b += sizeof(float) * QCmax + sizeof(int) * QCmax;    // lse2, tq
  b += sizeof(float) * kRedTiles * 4 * 128;            // red
  b += sizeof(int) * kRedTiles * 128;                  // cnt
  b += sizeof(uint64_t) * (2 * NS + 2 * kSlots + 2) + 16;  // barriers, tmem slot, abort flag
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
  p += sizeof(float) * kRedTiles * 4 * 128;
  s.cnt = reinterpret_cast<int*>(p);
  p += sizeof(int) * kRedTiles * 128;
  s.bars = reinterpret_cast<uint64_t*>(p);
  p += sizeof(uint64_t) * (2 * NS + 2 * kSlots + 2);
  s.tmem_slot = reinterpret_cast<uint32_t*>(p);
  s.abort_flag = reinterpret_cast<int*>(p + 8);
  return s;
}

// Barrier addresses.
__device__ __forceinline__ uint32_t bar_full(const Smem& sm, int st) { return smem_u32(&sm.bars[st]); }
__device__ __forceinline__ uint32_t bar_empty(const Smem& sm, int NS, int st) { return smem_u32(&sm.bars[NS + st]); }
__device__ __forceinline__ uint32_t bar_tfull(const Smem& sm, int NS, int s) { return smem_u32(&sm.bars[2 * NS + s]); }
__device__ __forceinline__ uint32_t bar_tempty(const Smem& sm, int NS, int s) {
  return smem_u32(&sm.bars[2 * NS + kSlots + s]);
}
__device__ __forceinline__ uint32_t bar_qfull(const Smem& sm, int NS) { return smem_u32(&sm.bars[2 * NS + 2 * kSlots]); }
__device__ __forceinline__ uint32_t bar_fin(const Smem& sm, int NS) { return smem_u32(&sm.bars[2 * NS + 2 * kSlots + 1]); }

__device__ __forceinline__ void init_barriers(const Smem& sm, int NS) {
  for (int i = 0; i < NS; ++i) {
    mbar_init(bar_full(sm, i), 1);
    mbar_init(bar_empty(sm, NS, i), 1);
  }
  for (int s = 0; s < kSlots; ++s) {
    mbar_init(bar_tfull(sm, NS, s), 1);
    mbar_init(bar_tempty(sm, NS, s), kEpiWarps / 2);   // the eight warps of one pair drain a slot
  }
  mbar_init(bar_qfull(sm, NS), 1);
  mbar_init(bar_fin(sm, NS), 1);
  *sm.abort_flag = 0;
  fence_barrier_init();
}

// Unit schedule.  A unit is key tile i against group h (128 query rows in
// pass 1, 128 query columns in pass 2), h in [0, H).  Warpgroup pair P owns the
// units with h % 2 == P (with one group per tile: the tiles with i % 2 == P)
// and alternates between TMEM slots P and P + 2, so the MMA can fill a pair's
// next slot while the pair drains the current one.
struct UnitSlot {
  int pair, slot;
  uint32_t parity;   // phase parity of this use of the slot
};

__device__ __forceinline__ UnitSlot unit_slot(int i, int h, int H) {
  UnitSlot u;
  int k;   // how many units the owning pair had before this one
  if (H >= 2) {
    u.pair = h & 1;
    const int per_tile = u.pair == 0 ? (H + 1) / 2 : H / 2;
    k = i * per_tile + (h >> 1);
  } else {
    u.pair = i & 1;
    k = i >> 1;
  }
  u.slot = u.pair + 2 * (k & 1);
  u.parity = (k >> 1) & 1;
  return u;
}

// An epilogue warp is done reading a TMEM slot: order its loads before the
// arrival the MMA issuer waits for.
__device__ __forceinline__ void release_slot(const Smem& sm, int NS, int slot, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_tempty(sm, NS, slot));
}

// Wait until the MMA has filled `slot` for the use with phase parity `parity`;
// false (and the abort flag set) on a timeout or another role's abort.
__device__ __forceinline__ bool wait_slot(const ScoreArgs& a, const Smem& sm, int NS, int slot, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(sm.abort_flag)) return false;
  if (!mbar_wait(bar_tfull(sm, NS, slot), parity, kWaitLimit)) {
    set_status(a.status, UPF_ERR_TIMEOUT);
    *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
    return false;
  }
  tc_fence_after();
  return true;
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

// sum_j 2^(v[j] * sl - ref) over 32 values, with the affine step and the
// accumulation in packed fp32 pairs (measured: fewer FMA-pipe instructions
// than the scalar form, even with the moves that form the pairs).
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

// Pass-1 epilogue step: fold 32 logits of one query row (raw dot products;
// masked entries already -inf) into its running (m, Z), with m and the
// exponents in log2 units scaled by sl = scale * log2(e).  m is a reference
// point, not necessarily the exact maximum: the exponentials are taken against
// the current m while the chunk maximum is reduced alongside, and m moves only
// when the maximum grew by more than 8 (so every term stays below 2^8 and
// m + log2 Z is unchanged).
__device__ __forceinline__ void online_update32(const float (&v)[32], float sl, float& m, float& z) {
  float t[10];
#pragma unroll
  for (int j = 0; j < 10; ++j) t[j] = max3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
  const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]), u2 = max3(t[6], t[7], t[8]);
  const float u3 = max3(t[9], v[30], v[31]);
  const float mx = fmaxf(max3(u0, u1, u2), u3);
  if (m == -INFINITY) {            // first visible chunk of this row
    if (mx == -INFINITY) return;
    m = mx * sl;
    z = exp_sum32(v, sl, m);
    return;
  }
  float sum = exp_sum32(v, sl, m);
  const float mxs = mx * sl;
  if (mxs > m + 8.f) {
    // terms against the old reference are below 2^96 unless the jump is
    // larger; then they are recomputed against the new one
    sum = mxs > m + 96.f ? exp_sum32(v, sl, mxs) : sum * ex2_approx(m - mxs);
    z *= ex2_approx(m - mxs);
    m = mxs;
  }
  z += sum;
}

// Pass-2 epilogue step: acc += 2^(v * sl - lse2) for 16 query columns of one
// key; nlse points at -lse2 of those columns in shared memory (16-byte aligned).
// acc0/acc1 hold packed fp32 pairs.
__device__ __forceinline__ void normalised_sum16(const float (&v)[16], const float* nlse, float sl, uint64_t& acc0,
                                                 uint64_t& acc1) {
  const float4* l4 = reinterpret_cast<const float4*>(nlse);
  const uint64_t sl2 = pack2(sl, sl);
#pragma unroll
  for (int j = 0; j < 16; j += 4) {
    const float4 l = l4[j / 4];
    float a, b, c, d;
    unpack2(fma2(pack2(v[j], v[j + 1]), sl2, pack2(l.x, l.y)), a, b);
    unpack2(fma2(pack2(v[j + 2], v[j + 3]), sl2, pack2(l.z, l.w)), c, d);
    acc0 = add2(acc0, pack2(ex2_approx(a), ex2_approx(b)));
    acc1 = add2(acc1, pack2(ex2_approx(c), ex2_approx(d)));
  }
}

// The same near the causal edge / request end: only columns the key is visible to.
__device__ __forceinline__ void normalised_sum16_masked(const float (&v)[16], const float* nlse, const int* tq,
                                                        int key, float sl, float& accm) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (key <= tq[j]) accm += ex2_approx(fmaf(v[j], sl, nlse[j]));
}

// One warp's share of a pass-1 unit: two chunks of 32 key columns of one
// query row at taddr.  Chunk 1 is loaded while chunk 0 is reduced; the slot is
// released as soon as chunk 1 has landed.  col0: first key column of this
// share inside the tile; t_row: the row's query position (-1: no row).
__device__ __forceinline__ void pass1_unit(uint32_t taddr, int col0, int kt, bool masked, int t_row, float sl,
                                           float& m, float& z, const Smem& sm, int NS, int slot, int lane) {
  float va[32], vb[32];
  tmem_ld32(taddr, va);
  tmem_wait_ld();
  tmem_ld32(taddr + 32u, vb);
  const int lim = t_row - kt - col0;   // columns j > lim of the share are invisible
  if (masked) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j > lim) va[j] = -INFINITY;
  }
  online_update32(va, sl, m, z);
  tmem_wait_ld();
  release_slot(sm, NS, slot, lane);
  if (masked) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j + 32 > lim) vb[j] = -INFINITY;
  }
  online_update32(vb, sl, m, z);
}

// One warp's share of a pass-2 unit: 64 query columns of one key, streamed
// from TMEM in four 16-column pieces through two register buffers (piece p+1
// loads while piece p is summed); the slot is released after the last load.
// nlse / tq point at the share's first column (-lse2 and query position).
__device__ __forceinline__ void pass2_unit(uint32_t taddr, const float* nlse, const int* tq, int key, bool masked,
                                           float sl, uint64_t& acc0, uint64_t& acc1, float& accm, const Smem& sm,
                                           int NS, int slot, int lane) {
  float v0[16], v1[16];
  auto sum = [&](const float (&v)[16], int c) {
    if (!masked) normalised_sum16(v, nlse + c, sl, acc0, acc1);
    else normalised_sum16_masked(v, nlse + c, tq + c, key, sl, accm);
  };
  tmem_ld16(taddr, v0);
  tmem_wait_ld();
  tmem_ld16(taddr + 16u, v1);
  sum(v0, 0);
  tmem_wait_ld();
  tmem_ld16(taddr + 32u, v0);
  sum(v1, 16);
  tmem_wait_ld();
  tmem_ld16(taddr + 48u, v1);
  sum(v0, 32);
  tmem_wait_ld();
  release_slot(sm, NS, slot, lane);
  sum(v1, 48);
}

// Producer: Q chunk (once), then key tiles slice by slice through the ring.
// Returns the number of key-slice loads issued.
__device__ int produce(const ScoreArgs& a, const CUtensorMap* tq_map, const CUtensorMap* tk_map, const Smem& sm,
                       const ItemTC& it, const ChunkShape& cs, int k0, int ntiles, int NS) {
  const int S = a.d / 64;
  // Query rows: boxes of BQ rows of one head.
  const int BQ = a.q_box_rows;
  const int boxes = cs.rows_c / BQ;
  mbar_arrive_expect_tx(bar_qfull(sm, NS), uint32_t(boxes) * S * BQ * 128);
  for (int b = 0; b < boxes; ++b) {
    const int rho = it.qc * a.QC + b * BQ;
    const int h = a.qhead[it.g * a.gamma + rho / a.n];
    const int tok = it.tok0 + it.L - a.n + rho % a.n;   // may be < 0 or in another request; masked later
    for (int s = 0; s < S; ++s)
      tma_load_3d(smem_u32(sm.q + size_t(s) * a.QC * 128 + size_t(b) * BQ * 128), tq_map, s * 64, h, tok,
                  bar_qfull(sm, NS));
  }
  int iter = 0;
  for (int i = 0; i < ntiles; ++i) {
    for (int s = 0; s < S; ++s, ++iter) {
      const int st = iter % NS;
      const uint32_t ph = (iter / NS) & 1;
      if (*reinterpret_cast<volatile int*>(sm.abort_flag)) return iter;
      if (!mbar_wait(bar_empty(sm, NS, st), ph ^ 1, kWaitLimit)) {
        set_status(a.status, UPF_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
        return iter;
      }
      mbar_arrive_expect_tx(bar_full(sm, st), kSliceBytes);
      tma_load_3d(smem_u32(sm.stages + size_t(st) * kSliceBytes), tk_map, s * 64, it.g, it.tok0 + k0 + i * kTile,
                  bar_full(sm, st));
    }
  }
  return iter;
}

// After an abort: wait (bounded) for the query load and for the last key
// load issued into each stage, so no copy is still landing when the CTA exits.
__device__ void drain_loads(const Smem& sm, int NS, int issued) {
  mbar_wait(bar_qfull(sm, NS), 0, kWaitLimit / 8);
  for (int st = 0; st < NS; ++st) {
    const int c = issued > st ? (issued - st + NS - 1) / NS : 0;   // loads issued into stage st
    if (c > 0) mbar_wait(bar_full(sm, st), (c - 1) & 1, kWaitLimit / 8);
  }
}

// One thread issues every unit's MMAs in order (M = N = 128, K = d).
// keys_as_m: pass 2 (A = key tile, B = query group); else pass 1 (A = query
// group, B = key tile).  Before returning it waits for all of them to finish.
__device__ void issue_mma(const ScoreArgs& a, const Smem& sm, int NS, int ntiles, int H, uint32_t tmem,
                          bool keys_as_m) {
  const int S = a.d / 64;
  const uint32_t idesc = idesc_bf16_f32(128, 128);
  bool ok = mbar_wait(bar_qfull(sm, NS), 0, kWaitLimit);
  int iter = 0;
  for (int i = 0; ok && i < ntiles; ++i) {
    for (int s = 0; s < S && ok; ++s) ok = mbar_wait(bar_full(sm, (iter + s) % NS), ((iter + s) / NS) & 1, kWaitLimit);
    if (!ok) break;
    tc_fence_after();
    for (int h = 0; h < H && ok; ++h) {
      const UnitSlot us = unit_slot(i, h, H);
      ok = mbar_wait(bar_tempty(sm, NS, us.slot), us.parity ^ 1, kWaitLimit);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dt = tmem + uint32_t(us.slot * 128);
      for (int s = 0; s < S; ++s) {
        const uint32_t kb = smem_u32(sm.stages + size_t((iter + s) % NS) * kSliceBytes);
        const uint32_t qg = smem_u32(sm.q + size_t(s) * a.QC * 128 + size_t(h) * 128 * 128);
        const uint32_t am = keys_as_m ? kb : qg, bn = keys_as_m ? qg : kb;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(dt, sdesc_kmajor_sw128(am + kk * 32), sdesc_kmajor_sw128(bn + kk * 32), idesc, (s | kk) ? 1u : 0u);
      }
      mma_commit(bar_tfull(sm, NS, us.slot));
    }
    for (int s = 0; s < S; ++s) mma_commit(bar_empty(sm, NS, (iter + s) % NS));
    iter += S;
  }
  if (!ok) {
    set_status(a.status, UPF_ERR_TIMEOUT);
    *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
  }
  // Every MMA this thread issued must be done before TMEM can be freed.
  mma_commit(bar_fin(sm, NS));
  mbar_wait(bar_fin(sm, NS), 0, kWaitLimit);
}

// Zero the padding rows [rows_c, QCp) of the query chunk (generic stores,
// ordered before any MMA reads by the caller's proxy fence + barrier).
__device__ __forceinline__ void zero_padding(const ScoreArgs& a, const Smem& sm, const ChunkShape& cs) {
  for (int s = 0; s < a.d / 64; ++s) {
    uint4* base = reinterpret_cast<uint4*>(sm.q + size_t(s) * a.QC * 128 + size_t(cs.rows_c) * 128);
    const int n16 = (cs.QCp - cs.rows_c) * 8;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
  }
}

// ------------------------------------------------------------- pass 1 -----

__global__ void __launch_bounds__(kThreadsTC, 1)
    score_pass1_tc(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                   const __grid_constant__ ScoreArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x;
  if (item >= a.items1 || item >= a.item_off1[a.R]) return;
  const int NS = stages_for(a.d);
  const Smem sm = carve(smem_raw, a.d, a.QC);
  const ItemTC it = locate_tc(a.item_off1, a.cu, a.R, item, a.KS1, a.NQC);
  const ChunkShape cs = chunk_shape(a, it.qc);
  const int k0 = it.s * a.KS1, k1 = min(it.L, k0 + a.KS1);
  const int ntiles = ceil_div_dev(k1 - k0, kTile);
  const int MT = cs.QCp / 128;            // M tiles (groups) of 128 query rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) init_barriers(sm, NS);
  zero_padding(a, sm, cs);
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
    if (lane == 0) issue_mma(a, sm, NS, ntiles, MT, tmem, false);
  } else {
    // Epilogue: pair P (warpgroups 2P, 2P+1) owns M tiles P and P+2 (with one
    // M tile: alternate key tiles); the pair's two warpgroups split each
    // unit's 128 key columns, so every thread keeps (m, Z) for up to two rows.
    const int wg = warp >> 2, qd = warp & 3;
    const int pair = wg >> 1, wsub = wg & 1;
    const int mrow = qd * 32 + lane;
    const int mt0 = MT >= 2 ? pair : 0, mt1 = pair + 2;
    const int row0 = mt0 * 128 + mrow, row1 = mt1 * 128 + mrow;
    const int t_row0 = (mt0 < MT && row0 < cs.rows_c) ? it.L - a.n + (it.qc * a.QC + row0) % a.n : -1;
    const int t_row1 = (MT >= 2 && mt1 < MT && row1 < cs.rows_c) ? it.L - a.n + (it.qc * a.QC + row1) % a.n : -1;
    const int col0 = wsub * 64;
    const float sl = a.scale_log2;
    float m0 = -INFINITY, z0 = 0.f, m1 = -INFINITY, z1 = 0.f;
    bool ok = true;
    for (int i = 0; ok && i < ntiles; ++i) {
      const int kt = k0 + i * kTile;
      const bool masked = kt + kTile - 1 > it.L - a.n;
      for (int h = 0; h < MT; ++h) {
        const UnitSlot us = unit_slot(i, h, MT);
        if (us.pair != pair) continue;
        if (!wait_slot(a, sm, NS, us.slot, us.parity)) {
          ok = false;
          break;
        }
        const uint32_t taddr = tmem + (uint32_t(qd * 32) << 16) + uint32_t(us.slot * 128 + col0);
        if (MT < 2 || (h >> 1) == 0) pass1_unit(taddr, col0, kt, masked, t_row0, sl, m0, z0, sm, NS, us.slot, lane);
        else pass1_unit(taddr, col0, kt, masked, t_row1, sl, m1, z1, sm, NS, us.slot, lane);
      }
    }
    // Merge the (m, Z) of the warpgroups that covered the same row, store.
    float2* red = reinterpret_cast<float2*>(sm.red);   // [4 wg][2][128]
    epi_bar();
    red[(wg * 2 + 0) * 128 + mrow] = make_float2(m0, z0);
    red[(wg * 2 + 1) * 128 + mrow] = make_float2(m1, z1);
    epi_bar();
    for (int j = 0; j < 2; ++j) {
      int mt, w_lo, w_hi;
      if (MT >= 2) {
        if (wsub != 0) break;
        mt = pair + 2 * j;
        w_lo = 2 * pair;
        w_hi = 2 * pair + 1;
      } else {
        if (wg != 0 || j != 0) break;
        mt = 0;
        w_lo = 0;
        w_hi = 3;
      }
      const int row = mt * 128 + mrow;
      if (mt >= MT || row >= cs.rows_c) continue;
      float mm = -INFINITY;
      for (int w = w_lo; w <= w_hi; ++w) mm = fmaxf(mm, red[(w * 2 + j) * 128 + mrow].x);
      float zz = 0.f;
      if (mm > -INFINITY)
        for (int w = w_lo; w <= w_hi; ++w) {
          const float2 p = red[(w * 2 + j) * 128 + mrow];
          if (p.y > 0.f) zz += p.y * ex2_approx(p.x - mm);
        }
      a.p1part[(int64_t)item * a.QC + row] = make_float2(mm, zz);
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
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x;
  if (item >= a.items2 || item >= a.item_off2[a.R]) return;
  const int NS = stages_for(a.d);
  const Smem sm = carve(smem_raw, a.d, a.QC);
  const ItemTC it = locate_tc(a.item_off2, a.cu, a.R, item, a.KS2, a.NQC);
  const ChunkShape cs = chunk_shape(a, it.qc);
  const int k0 = it.s * a.KS2, k1 = min(it.L, k0 + a.KS2);
  const int ntiles = ceil_div_dev(k1 - k0, kTile);
  const int H = cs.QCp / 128;             // groups of 128 query columns
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) init_barriers(sm, NS);
  zero_padding(a, sm, cs);
  for (int i = tid; i < kRedTiles * 128; i += blockDim.x) sm.cnt[i] = 0;
  // lse2 of every query row of the chunk from the pass-1 partials, stored
  // negated; -inf marks rows that do not exist (padding, or positions before
  // the request start).
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
      sm.lse2[row] = -l2;
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
    if (lane == 0) issue_mma(a, sm, NS, ntiles, H, tmem, true);
  } else {
    // Epilogue: pair P owns the groups h with h % 2 == P (with one group:
    // alternate key tiles); the pair's two warpgroups split each unit's 128
    // query columns.  Per key tile the warpgroup sums for a key are combined
    // without a barrier: the last to arrive adds them in a fixed order.
    const int wg = warp >> 2, qd = warp & 3;
    const int pair = wg >> 1, wsub = wg & 1;
    const int krow = qd * 32 + lane;
    const float sl = a.scale_log2;
    float* out = a.part + (int64_t)(it.g * a.NQC + it.qc) * a.T + it.tok0;
    const int expect = H >= 2 ? 4 : 2;
    bool ok = true;
    for (int i = 0; ok && i < ntiles; ++i) {
      const int kt = k0 + i * kTile;
      const int key = kt + krow;
      const bool masked = kt + kTile - 1 > it.L - a.n;
      uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);
      float accm = 0.f;
      bool mine = false;
      for (int h = 0; h < H; ++h) {
        const UnitSlot us = unit_slot(i, h, H);
        if (us.pair != pair) continue;
        if (!wait_slot(a, sm, NS, us.slot, us.parity)) {
          ok = false;
          break;
        }
        const int col0 = h * 128 + wsub * 64;
        const uint32_t taddr = tmem + (uint32_t(qd * 32) << 16) + uint32_t(us.slot * 128 + wsub * 64);
        pass2_unit(taddr, sm.lse2 + col0, sm.tq + col0, key, masked, sl, acc0, acc1, accm, sm, NS, us.slot, lane);
        mine = true;
      }
      if (!ok || !mine) continue;
      float lo, hi;
      unpack2(add2(acc0, acc1), lo, hi);
      volatile float* red = sm.red + (i % kRedTiles) * 512;
      int* cnt = sm.cnt + (i % kRedTiles) * 128;
      red[wg * 128 + krow] = (lo + hi) + accm;
      __threadfence_block();
      if (atomicAdd(&cnt[krow], 1) == expect - 1) {
        __threadfence_block();
        const float tot = H >= 2 ? ((red[krow] + red[128 + krow]) + red[256 + krow]) + red[384 + krow]
                                 : red[(2 * pair) * 128 + krow] + red[(2 * pair + 1) * 128 + krow];
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

cudaError_t launch_score_pass1_tc(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  if (a.items1 == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.d, a.Hq, a.T, a.q_stride, a.q_box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.d, a.Hkv, a.T, a.k_stride, kTile)) != cudaSuccess) return e;
  const size_t smem = smem_bytes_tc(a.d, a.QC);
  if ((e = cudaFuncSetAttribute(score_pass1_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
    return e;
  return launch_kernel(score_pass1_tc, a.items1, kThreadsTC, smem, s, pdl, mq, mk, a);
}

cudaError_t launch_score_pass2_tc(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  if (a.items2 == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.d, a.Hq, a.T, a.q_stride, a.q_box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.d, a.Hkv, a.T, a.k_stride, kTile)) != cudaSuccess) return e;
  const size_t smem = smem_bytes_tc(a.d, a.QC);
  if ((e = cudaFuncSetAttribute(score_pass2_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
    return e;
  return launch_kernel(score_pass2_tc, a.items2, kThreadsTC, smem, s, pdl, mq, mk, a);
}

}  // namespace upf
