// Tensor-core scoring passes on CTA pairs (tcgen05.mma.cta_group::2), sm_103a.
//
// UniPrefill article, section 二 first step (the last n tokens score every
// token) and section 三 (scores and their online normalisation on the GPU):
// the same two passes as score_tc.cu, but each work item runs on a cluster of
// two CTAs on two SMs that share one M = 256 MMA:
//
//   pass 1 (queries on M): a 256-row query unit (rows 0-127 in CTA 0's shared
//     memory, 128-255 in CTA 1's) against a 256-key tile (keys 0-127 from CTA
//     0, 128-255 from CTA 1); each CTA's TMEM receives its 128 query rows by
//     256 keys, and its epilogue keeps their running (m, Z);
//   pass 2 (keys on M): a 256-key tile (128 keys per CTA) against a 256-column
//     query unit (128 columns per CTA); each CTA's TMEM receives its 128 keys
//     by 256 query columns, and its epilogue sums the normalised terms.
//
// Compared with one CTA per item, each SM holds half of the query chunk (a
// deeper key ring fits) and the tensor core reads 8 instead of 12 KB of
// shared memory per 128 clocks.  Each CTA loads its own halves with TMA into
// its own ring (no multicast) and waits for its own copies; CTA 1's otherwise
// idle MMA warp relays each landed stage to CTA 0 with a remote mbarrier
// arrive, and CTA 0's MMA thread issues the MMAs once both halves are there.
// Completion commits are multicast to both CTAs; CTA 1's epilogue warps hand
// accumulator slots back to CTA 0 with remote arrives.  TMEM is allocated and
// freed by one warp of each CTA together.  Every wait is bounded; a timeout
// in either CTA aborts both (the flag is written into the peer too), both
// wind down, wait for their own copies and for the MMAs, meet at a cluster
// barrier and free TMEM.
#include "score_common.cuh"
#include "sm100_ptx.cuh"
#include "upf_internal.cuh"

#ifndef UPF_PAIR_SLOTS
#define UPF_PAIR_SLOTS 2
#endif

namespace upf {

namespace {

static_assert(UPF_PAIR_SLOTS == 1 || UPF_PAIR_SLOTS == 2, "one or two 256-column accumulator slots");
constexpr int kW = 4;                          // epilogue warps per TMEM lane quarter
constexpr int kEpiWarps = 4 * kW;              // 16
constexpr int kEpiThreads = kEpiWarps * 32;    // 512
constexpr int kProducerWarp = kEpiWarps;       // 16
constexpr int kMmaWarp = kEpiWarps + 1;        // 17: MMA issuer in CTA 0, relay in CTA 1
constexpr int kThreadsPair = kEpiThreads + 64; // 576
constexpr int kHalf = 128;                     // M rows and N columns each CTA supplies
constexpr int kPairTile = 256;                 // keys per tile of the pair
constexpr int kStageBytes = 32768;
constexpr int kMaxStages = 8;
constexpr int kSlots = UPF_PAIR_SLOTS;         // TMEM accumulator slots of 256 columns
constexpr uint32_t kTmemCols = 256u * kSlots;
constexpr int kRedTiles = 8;
// full[8], peer_full[8], empty[8], tfull[2], tempty[2], qfull, peer_qfull, fin
constexpr int kNumBars = 3 * kMaxStages + 2 * kSlots + 3;
constexpr int kSmemLimit = 232448;
constexpr long long kWaitLimit = kDefaultWaitCycles;
constexpr uint32_t kIdleNs = 4000;
constexpr uint32_t kRemoteNs = 64;   // polls of phases that the peer CTA completes

struct PGeo {
  int S;            // 64-wide slices of the head dim
  int slice_bytes;  // 128 rows x 128 B
  int sps;          // slices per ring stage
  int spt;          // ring stages per tile
  int stage_bytes;
  int U;            // 256-wide query units of a full chunk
  int q_bytes;      // this CTA's half of the query chunk: S slices x U*128 rows x 128 B
  int extra_bytes;  // pass 2: -lse2 and positions of the chunk's columns, per-key partial sums
  int NS;           // ring stages
  int smem;
};

__host__ __device__ inline PGeo pair_geometry(int pass, int d, int QC) {
  PGeo g;
  g.S = d / 64;
  g.slice_bytes = kHalf * 128;
  g.sps = imax(1, imin(g.S, kStageBytes / g.slice_bytes));
  g.spt = g.S / g.sps;
  g.stage_bytes = g.sps * g.slice_bytes;
  g.U = QC / 256;
  g.q_bytes = g.S * g.U * kHalf * 128;
  g.extra_bytes = pass == 2 ? 8 * QC + kRedTiles * kW * 128 * 4 : 0;
  const int fixed = 1024 /* alignment slack */ + g.q_bytes + g.extra_bytes + 8 * kNumBars + 16;
  g.NS = imin(kMaxStages, (kSmemLimit - fixed) / g.stage_bytes);
  g.smem = fixed + g.NS * g.stage_bytes;
  return g;
}

struct PSmem {
  unsigned char* q;     // S slices x (U*128) rows x 128 B, 1024-aligned
  unsigned char* ring;  // NS stages
  float* nlse;          // pass 2: -lse2 per chunk column
  int* tq;              // pass 2: query position per chunk column (-1: none)
  float* red;           // pass 2: [kRedTiles][kW][128] per-key sums of the column quarters
  uint64_t* bars;
  uint32_t* tmem_slot;
  int* abort_flag;
};

__device__ __forceinline__ PSmem pcarve(unsigned char* raw, const PGeo& g, int QC) {
  PSmem s;
  unsigned char* p = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.q = p;
  p += g.q_bytes;
  s.ring = p;
  p += g.NS * g.stage_bytes;
  s.nlse = reinterpret_cast<float*>(p);
  s.tq = reinterpret_cast<int*>(p + 4 * QC);
  s.red = reinterpret_cast<float*>(p + 8 * QC);
  p += g.extra_bytes;
  s.bars = reinterpret_cast<uint64_t*>(p);
  p += 8 * kNumBars;
  s.tmem_slot = reinterpret_cast<uint32_t*>(p);
  s.abort_flag = reinterpret_cast<int*>(p + 8);
  return s;
}

__device__ __forceinline__ uint32_t b_full(const PSmem& sm, int st) { return smem_u32(&sm.bars[st]); }
__device__ __forceinline__ uint32_t b_pfull(const PSmem& sm, int st) { return smem_u32(&sm.bars[kMaxStages + st]); }
__device__ __forceinline__ uint32_t b_empty(const PSmem& sm, int st) { return smem_u32(&sm.bars[2 * kMaxStages + st]); }
__device__ __forceinline__ uint32_t b_tfull(const PSmem& sm, int s) { return smem_u32(&sm.bars[3 * kMaxStages + s]); }
__device__ __forceinline__ uint32_t b_tempty(const PSmem& sm, int s) {
  return smem_u32(&sm.bars[3 * kMaxStages + kSlots + s]);
}
__device__ __forceinline__ uint32_t b_qfull(const PSmem& sm) { return smem_u32(&sm.bars[3 * kMaxStages + 2 * kSlots]); }
__device__ __forceinline__ uint32_t b_pqfull(const PSmem& sm) {
  return smem_u32(&sm.bars[3 * kMaxStages + 2 * kSlots + 1]);
}
__device__ __forceinline__ uint32_t b_fin(const PSmem& sm) { return smem_u32(&sm.bars[3 * kMaxStages + 2 * kSlots + 2]); }

__device__ __forceinline__ bool paborted(const PSmem& sm) { return *reinterpret_cast<volatile int*>(sm.abort_flag) != 0; }

// Record a timeout and stop both CTAs of the pair.
__device__ __forceinline__ void pabort(const ScoreArgs& a, const PSmem& sm, uint32_t rank) {
  set_status(a.status, UPF_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
  st_cluster_u32(mapa_shared(smem_u32(sm.abort_flag), rank ^ 1u), 1u);
}

__device__ __forceinline__ int chunk_rows_p(const ScoreArgs& a, int qc) { return min(a.QC, a.QR - qc * a.QC); }

// Local query row lr (unit lr / 128, row lr % 128 of this CTA's half) is row
// 256 u + 128 rank + r of the chunk.
__device__ __forceinline__ int chunk_row_of(int lr, uint32_t rank) { return (lr >> 7) * 256 + int(rank) * kHalf + (lr & 127); }

// Barriers, zeroed padding rows of this CTA's query half, the pair's TMEM,
// and a cluster barrier (the peer's barriers exist before anything signals
// them).  Returns the TMEM base.
__device__ uint32_t pair_setup(const ScoreArgs& a, const PSmem& sm, const PGeo& geo, int rows_c, uint32_t rank) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(b_full(sm, i), 1);
      mbar_init(b_pfull(sm, i), 1);
      mbar_init(b_empty(sm, i), 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(b_tfull(sm, s), 1);
      mbar_init(b_tempty(sm, s), 2 * kEpiWarps);   // both CTAs' epilogue warps drain every unit
    }
    mbar_init(b_qfull(sm), 1);
    mbar_init(b_pqfull(sm), 1);
    mbar_init(b_fin(sm), 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  // rows of this CTA's half that lie past the chunk's end are zero
  const int rows_local = geo.U * kHalf;
  for (int s = 0; s < geo.S; ++s) {
    unsigned char* base = sm.q + size_t(s) * rows_local * 128;
    for (int i = threadIdx.x; i < rows_local * 8; i += blockDim.x) {
      const int lr = i >> 3;
      if (chunk_row_of(lr, rank) >= rows_c) reinterpret_cast<uint4*>(base + size_t(lr) * 128)[i & 7] = make_uint4(0, 0, 0, 0);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(sm.tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  return *sm.tmem_slot;
}

// Producer (one lane): this CTA's half of the query chunk, then its 128 keys
// of every pair tile, stage by stage.  Returns the stage loads issued.
template <bool kDescending>
__device__ int pair_produce(const ScoreArgs& a, const CUtensorMap* tq_map, const CUtensorMap* tk_map, const PSmem& sm,
                            const PGeo& geo, const ItemTC& it, int rows_c, int U, int k0, int ntiles, uint32_t rank) {
  const int BQ = a.q_box_rows;
  const int rows_local = geo.U * kHalf;
  int boxes = 0;
  for (int lr = 0; lr < U * kHalf; lr += BQ)
    if (chunk_row_of(lr, rank) < rows_c) ++boxes;
  mbar_arrive_expect_tx(b_qfull(sm), uint32_t(boxes) * geo.S * BQ * 128);
  for (int lr = 0; lr < U * kHalf; lr += BQ) {
    const int row = chunk_row_of(lr, rank);
    if (row >= rows_c) continue;
    const int rho = it.qc * a.QC + row;
    const int h = a.qhead[it.g * a.gamma + rho / a.n];
    const int tok = it.tok0 + it.L - a.n + rho % a.n;   // may be < 0 or in another request; masked later
    for (int s = 0; s < geo.S; ++s)
      tma_load_3d(smem_u32(sm.q + size_t(s) * rows_local * 128 + size_t(lr) * 128), tq_map, s * 64, h, tok,
                  b_qfull(sm));
  }
  const int total = ntiles * geo.spt;
  int q = 0, st = 0, part = 0;
  uint32_t ph = 0;
  int key = it.tok0 + k0 + int(rank) * kHalf + (kDescending ? (ntiles - 1) * kPairTile : 0);
  for (int n = 0; n < total; ++n, ++q) {
    if (paborted(sm)) return q;
    if (!mbar_wait_idle(b_empty(sm, st), ph ^ 1u, a.wait_limit, kIdleNs)) {
      pabort(a, sm, rank);
      return q;
    }
    const uint32_t dst = smem_u32(sm.ring) + uint32_t(st * geo.stage_bytes);
    mbar_arrive_expect_tx(b_full(sm, st), uint32_t(geo.stage_bytes));
    for (int ss = 0; ss < geo.sps; ++ss)
      tma_load_3d(dst + uint32_t(ss * geo.slice_bytes), tk_map, (part * geo.sps + ss) * 64, it.g, key, b_full(sm, st));
    if (++st == geo.NS) { st = 0; ph ^= 1u; }
    if (++part == geo.spt) { part = 0; key += kDescending ? -kPairTile : kPairTile; }
  }
  return q;
}

// After an abort: wait (bounded) for this CTA's query load and for the last
// key load issued into each stage.
__device__ void pair_drain(const PSmem& sm, const PGeo& geo, int issued) {
  mbar_wait(b_qfull(sm), 0, kWaitLimit / 8);
  for (int st = 0; st < geo.NS; ++st) {
    const int c = issued > st ? (issued - st + geo.NS - 1) / geo.NS : 0;
    if (c > 0) mbar_wait(b_full(sm, st), (c - 1) & 1, kWaitLimit / 8);
  }
}

// CTA 1's MMA warp lane: tell CTA 0 about every one of this CTA's loads once
// it has landed, in issue order.
__device__ void pair_relay(const ScoreArgs& a, const PSmem& sm, const PGeo& geo, int ntiles) {
  if (!mbar_wait_idle(b_qfull(sm), 0, a.wait_limit, kIdleNs)) {
    pabort(a, sm, 1);
    return;
  }
  mbar_arrive_remote(mapa_shared(b_pqfull(sm), 0));
  const int total = ntiles * geo.spt;
  int st = 0;
  uint32_t ph = 0;
  for (int n = 0; n < total; ++n) {
    if (paborted(sm)) return;
    if (!mbar_wait_idle(b_full(sm, st), ph, a.wait_limit, kIdleNs)) {
      pabort(a, sm, 1);
      return;
    }
    mbar_arrive_remote(mapa_shared(b_pfull(sm, st), 0));
    if (++st == geo.NS) { st = 0; ph ^= 1u; }
  }
}

// CTA 0's MMA thread.  keys_as_m: pass 2 (A = key stage, B = query unit);
// else pass 1 (A = query unit, B = key stage).
template <bool kEarly>
__device__ void pair_mma(const ScoreArgs& a, const PSmem& sm, const PGeo& geo, int ntiles, int U, uint32_t tmem,
                         bool keys_as_m) {
  const uint32_t idesc = idesc_bf16_f32(256, 256);
  const uint32_t ring0 = smem_u32(sm.ring), q0 = smem_u32(sm.q);
  const uint32_t q_slice = uint32_t(geo.U * kHalf) * 128u;
  const uint32_t q_unit = uint32_t(kHalf) * 128u;
  bool ok = mbar_wait_idle(b_qfull(sm), 0, a.wait_limit, kIdleNs) &&
            mbar_wait_cluster(b_pqfull(sm), 0, a.wait_limit, kRemoteNs);
  int st = 0, slot = 0;
  uint32_t ph = 0, sph = 0;
  for (int i = 0; ok && i < ntiles; ++i) {
    if (paborted(sm)) {
      ok = false;
      break;
    }
    // Pass 2 (kEarly) with two stages per tile: the tile's first unit starts
    // on the first stage while the second may still be landing, and the first
    // stage is released as soon as the last unit has read it (as in the
    // single-CTA kernels).  Measured faster in pass 2 and slower in pass 1,
    // where the release is a commit in the middle of the tile's only unit.
    const int st0 = st, st1 = st + 1 == geo.NS ? 0 : st + 1;
    const uint32_t ph1 = st1 == 0 ? ph ^ 1u : ph;
    const bool two = kEarly && geo.spt == 2;
    ok = mbar_wait_idle(b_full(sm, st0), ph, a.wait_limit, kIdleNs) &&
         mbar_wait_cluster(b_pfull(sm, st0), ph, a.wait_limit, kRemoteNs);
    if (!kEarly && ok && geo.spt == 2)
      ok = mbar_wait_idle(b_full(sm, st1), ph1, a.wait_limit, kIdleNs) &&
           mbar_wait_cluster(b_pfull(sm, st1), ph1, a.wait_limit, kRemoteNs);
    if (geo.spt == 2) { st = st1 + 1 == geo.NS ? 0 : st1 + 1; ph = (st1 == 0 || st == 0) ? ph ^ 1u : ph; }
    else { st = st1; ph = st1 == 0 ? ph ^ 1u : ph; }
    if (!ok) break;
    tc_fence_after();
    const uint32_t k0a = ring0 + uint32_t(st0 * geo.stage_bytes), k1a = ring0 + uint32_t(st1 * geo.stage_bytes);
    for (int u = 0; u < U; ++u) {
      ok = mbar_wait_cluster(b_tempty(sm, slot), sph ^ 1u, a.wait_limit, kRemoteNs);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dt = tmem + uint32_t(slot * 256);
      const uint32_t qu = q0 + uint32_t(u) * q_unit;
      for (int s = 0; s < geo.S; ++s) {
        if (kEarly && two && s == geo.sps) {   // the first slice of the second stage
          if (u == U - 1) mma_commit_pair_mc(b_empty(sm, st0), 0x3);
          if (u == 0) {
            ok = mbar_wait_idle(b_full(sm, st1), ph1, a.wait_limit, kIdleNs) &&
                 mbar_wait_cluster(b_pfull(sm, st1), ph1, a.wait_limit, kRemoteNs);
            if (!ok) break;
            tc_fence_after();
          }
        }
        const int part = geo.sps == 2 ? (s >> 1) : s;
        const uint32_t kb = (part == 0 ? k0a : k1a) + uint32_t(geo.sps == 2 ? (s & 1) * geo.slice_bytes : 0);
        const uint32_t qb = qu + uint32_t(s) * q_slice;
        const uint64_t da = sdesc_kmajor_sw128(keys_as_m ? kb : qb);
        const uint64_t db = sdesc_kmajor_sw128(keys_as_m ? qb : kb);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // +32 bytes along K = +2 in the descriptors' address field
          mma_bf16_pair(dt, da + uint64_t(2 * kk), db + uint64_t(2 * kk), idesc, (s | kk) ? 1u : 0u);
      }
      if (kEarly && !ok) break;
      mma_commit_pair_mc(b_tfull(sm, slot), 0x3);
      if (++slot == kSlots) { slot = 0; sph ^= 1u; }
    }
    if (!ok) break;
    if (!kEarly) {
      mma_commit_pair_mc(b_empty(sm, st0), 0x3);
      if (geo.spt == 2) mma_commit_pair_mc(b_empty(sm, st1), 0x3);
    } else {
      mma_commit_pair_mc(b_empty(sm, two ? st1 : st0), 0x3);
    }
  }
  if (!ok) pabort(a, sm, 0);
  // Every MMA issued must be done before either CTA frees TMEM (full limit).
  mma_commit_pair_mc(b_fin(sm), 0x1);
  if (!mbar_wait_idle(b_fin(sm), 0, kWaitLimit, kIdleNs)) pabort(a, sm, 0);
}

// An epilogue warp is done reading a TMEM slot: CTA 0's MMA thread waits for
// all 32 warps of the pair.
__device__ __forceinline__ void pair_release(const PSmem& sm, int slot, int lane, uint32_t rank) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (rank == 0) mbar_arrive(b_tempty(sm, slot));
    else mbar_arrive_remote(mapa_shared(b_tempty(sm, slot), 0));
  }
}

__device__ __forceinline__ bool pair_wait_slot(const ScoreArgs& a, const PSmem& sm, int slot, uint32_t parity,
                                               uint32_t rank) {
  if (mbar_try_wait(b_tfull(sm, slot), parity)) {
    tc_fence_after();
    return true;
  }
  if (paborted(sm)) return false;
  // CTA 1's slots are filled by CTA 0's multicast commit: short polls there.
  if (!mbar_wait_idle(b_tfull(sm, slot), parity, a.wait_limit, rank ? kRemoteNs : kIdleNs)) {
    pabort(a, sm, rank);
    return false;
  }
  tc_fence_after();
  return true;
}

__device__ __forceinline__ void pepi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

// Wind down: this CTA's outstanding loads after an abort, the pair meets,
// TMEM is freed by both CTAs together.
__device__ __forceinline__ void pair_teardown(const PSmem& sm, const PGeo& geo, int issued, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kProducerWarp && lane == 0 && paborted(sm)) pair_drain(sm, geo, issued);
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- pass 1 -----

// Epilogue of pass 1: this thread is row 32 qd + lane of this CTA's half of
// every query unit (MT = U <= 2 rows) and covers keys [64 cb, 64 cb + 64) of
// every 256-key tile.  Every unit's sums go through the checked online step
// (the reference m moves whenever a unit's sums leave [0, 2^20]).
__device__ void pair_pass1_epilogue(const ScoreArgs& a, const PSmem& sm, const ItemTC& it, int item, int rows_c,
                                    int U, int k0, int ntiles, uint32_t tmem, int warp, int lane, uint32_t rank) {
  const int qd = warp & 3, cb = warp >> 2;
  const float sl = a.scale_log2;
  const int r0 = qd * 32 + lane;
  auto lim_of = [&](int u) {   // last visible key of the row, relative to the tile start and this quarter
    const int row = u * 256 + int(rank) * kHalf + r0;
    return (u < U && row < rows_c) ? it.L - a.n + (it.qc * a.QC + row) % a.n - cb * 64 : INT_MIN;
  };
  const int l0 = lim_of(0), l1 = lim_of(1);
  float m0 = -INFINITY, m1 = -INFINITY, z0 = 0.f, z1 = 0.f;
  const uint32_t tbase = tmem + (uint32_t(qd * 32) << 16) + uint32_t(cb * 64);
  bool ok = true;
  int uidx = 0;
  for (int i = 0; ok && i < ntiles; ++i) {
    const int kt = k0 + i * kPairTile;
    const bool masked = kt + kPairTile - 1 > it.L - a.n;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u >= U) break;
      const int slot = uidx % kSlots;
      if (!pair_wait_slot(a, sm, slot, (uidx / kSlots) & 1, rank)) {
        ok = false;
        break;
      }
      ++uidx;
      const int lu = u == 0 ? l0 : l1;
      float mh = u == 0 ? m0 : m1;
      float zh = u == 0 ? z0 : z1;
      float va[32], vb[32];
      const uint32_t ta = tbase + uint32_t(slot * 256);
      tmem_ld32(ta, va);
      tmem_ld32(ta + 32u, vb);
      tmem_wait_ld();
      pair_release(sm, slot, lane, rank);
      if (lu != INT_MIN) {
        const int lim = lu - kt;   // this warp's columns j > lim are invisible
        if (masked) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j > lim) va[j] = -INFINITY;
            if (32 + j > lim) vb[j] = -INFINITY;
          }
        }
        const float sa = exp_sum32(va, sl, mh), sb = exp_sum32(vb, sl, mh);
        if (sa <= 1048576.f && sb <= 1048576.f) zh += sa + sb;
        else online_rescale<2>(va, vb, sl, mh, zh);
      }
      if (u == 0) { m0 = mh; z0 = zh; }
      else { m1 = mh; z1 = zh; }
    }
  }
  // Merge the four column quarters of every row through the (idle) ring.
  float2* red = reinterpret_cast<float2*>(sm.ring);   // [kW][U*128]
  const int rows_local = U * kHalf;
  if (ok) {
    red[cb * rows_local + r0] = make_float2(m0, z0);
    if (U > 1) red[cb * rows_local + kHalf + r0] = make_float2(m1, z1);
  }
  pepi_bar();
  if (!ok || paborted(sm)) return;
  for (int lr = cb * kHalf + r0; lr < rows_local; lr += kW * kHalf) {
    const int row = chunk_row_of(lr, rank);
    if (row >= rows_c) continue;
    float mm = -INFINITY;
#pragma unroll
    for (int c = 0; c < kW; ++c) mm = fmaxf(mm, red[c * rows_local + lr].x);
    float zz = 0.f;
    if (mm > -INFINITY) {
#pragma unroll
      for (int c = 0; c < kW; ++c) {
        const float2 p = red[c * rows_local + lr];
        if (p.y > 0.f) zz += p.y * ex2_approx(p.x - mm);
      }
    }
    a.p1part[(int64_t)item * a.QC + row] = make_float2(mm, zz);
  }
}

__global__ void __launch_bounds__(kThreadsPair, 1)
    score_pass1_pair(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                     const __grid_constant__ ScoreArgs a) {
  pdl_wait();      // then let pass 2 launch, which may read the queries and keys early
  pdl_trigger();
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x >> 1;
  const uint32_t rank = cluster_ctarank();
  if (!item_exists(a, item, false)) return;   // both CTAs of the pair alike
  const PGeo geo = pair_geometry(1, a.d, a.QC);
  const PSmem sm = pcarve(smem_raw, geo, a.QC);
  const ItemTC it = locate_item(a, item, false);
  const int rows_c = chunk_rows_p(a, it.qc);
  const int U = (rows_c + 255) / 256;
  const int k0 = it.s * a.KS1, k1 = min(it.L, k0 + a.KS1);
  const int ntiles = ceil_div_dev(k1 - k0, kPairTile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = pair_setup(a, sm, geo, rows_c, rank);
  int issued = 0;
  if (warp == kProducerWarp) {
    if (lane == 0) issued = pair_produce<false>(a, &tq_map, &tk_map, sm, geo, it, rows_c, U, k0, ntiles, rank);
    if (blockIdx.x == 0) desc_check(a, lane);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      if (rank == 0) pair_mma<false>(a, sm, geo, ntiles, U, tmem, false);
      else pair_relay(a, sm, geo, ntiles);
    }
  } else {
    pair_pass1_epilogue(a, sm, it, item, rows_c, U, k0, ntiles, tmem, warp, lane, rank);
  }
  pair_teardown(sm, geo, issued, tmem);
}

// ------------------------------------------------------------- pass 2 -----

// Epilogue of pass 2: this thread is key 128 rank + 32 qd + lane of every
// 256-key tile; its warp reads the 32-column chunks cb and cb + 4 of every
// unit and stores its per-key sum in red[i % kRedTiles][cb].  The quarter's
// first warp adds the kW sums of tile i - lag in a fixed order and writes
// them out (the slot hand-over orders those stores before the read, as in
// the one-CTA kernel).
__device__ void pair_pass2_epilogue(const ScoreArgs& a, const PSmem& sm, const ItemTC& it, int U, int k0, int k1,
                                    int ntiles, uint32_t tmem, int warp, int lane, uint32_t rank) {
  const int qd = warp & 3, cb = warp >> 2;
  const int krow = qd * 32 + lane;
  const float sl = a.scale_log2;
  float* out = a.part + (int64_t)(it.g * a.NQC + it.qc) * a.T + it.tok0;
  const uint32_t tq = tmem + (uint32_t(qd * 32) << 16) + uint32_t(cb * 32);
  // A warp holding unit x knows every warp released unit x - kSlots, hence
  // stored the sums of every tile before that unit's tile.
  const int lag = 1 + (kSlots + U - 1) / U;
  const uint32_t nlse_s = smem_u32(sm.nlse);
  bool ok = true;
  int uidx = 0;
  // Tiles run from the item's last keys to its first: pass 1 read the keys in
  // ascending order, so the last ones it read may still be in L2.
  const int klast = k0 + (ntiles - 1) * kPairTile + int(rank) * kHalf;   // this CTA's first key of the last tile
  for (int i = 0; i < ntiles; ++i) {
    const int kt = klast - i * kPairTile;   // this CTA's first key of the tile
    const int key = kt + krow;
    const bool masked = kt + kHalf - 1 > it.L - a.n;
    uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);
    for (int u = 0; u < U; ++u, ++uidx) {
      const int slot = uidx % kSlots;
      if (!pair_wait_slot(a, sm, slot, (uidx / kSlots) & 1, rank)) {
        ok = false;
        break;
      }
      if (u == 0 && cb == 0 && i >= lag) {   // tile i - lag is complete: write it out
        const int kprev = key + lag * kPairTile;
        if (kprev < k1) out[kprev] = [&] {
            const float* r = sm.red + ((i - lag) % kRedTiles) * kW * 128 + krow;
            float t = r[0];
#pragma unroll
            for (int c = 1; c < kW; ++c) t += r[c * 128];
            return t;
          }();
      }
      const int col0 = u * 256 + cb * 32;
      float va[32], vb[32];
      const uint32_t ta = tq + uint32_t(slot * 256);
      tmem_ld32(ta, va);
      tmem_ld32(ta + uint32_t(32 * kW), vb);
      tmem_wait_ld();
      pair_release(sm, slot, lane, rank);
      if (!masked) {
        normalised_sum32(va, nlse_s + 4 * col0, sl, acc0, acc1);
        normalised_sum32(vb, nlse_s + 4 * (col0 + 32 * kW), sl, acc0, acc1);
      } else {
        float t = normalised_sum32_masked(va, sm.nlse + col0, sm.tq + col0, key, sl);
        t += normalised_sum32_masked(vb, sm.nlse + col0 + 32 * kW, sm.tq + col0 + 32 * kW, key, sl);
        acc0 = add2(acc0, pack2(t, 0.f));
      }
    }
    if (!ok) break;
    float lo, hi;
    unpack2(add2(acc0, acc1), lo, hi);
    sm.red[((i % kRedTiles) * kW + cb) * 128 + krow] = lo + hi;
  }
  pepi_bar();
  if (ok && cb == 0 && !paborted(sm))
    for (int i = max(0, ntiles - lag); i < ntiles; ++i) {
      const int key = klast - i * kPairTile + krow;
      if (key < k1) {
        const float* r = sm.red + (i % kRedTiles) * kW * 128 + krow;
        float t = r[0];
#pragma unroll
        for (int c = 1; c < kW; ++c) t += r[c * 128];
        out[key] = t;
      }
    }
}

__global__ void __launch_bounds__(kThreadsPair, 1)
    score_pass2_pair(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                     const __grid_constant__ ScoreArgs a) {
  // As in the single-CTA pass 2: with the descriptor in the parameters only
  // the epilogue, which reads pass 1's partials, waits for pass 1.
  const bool early = a.desc.R > 0;
  pdl_trigger();
  if (!early) pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x >> 1;
  const uint32_t rank = cluster_ctarank();
  if (!item_exists(a, item, true)) return;   // both CTAs of the pair alike
  const PGeo geo = pair_geometry(2, a.d, a.QC);
  const PSmem sm = pcarve(smem_raw, geo, a.QC);
  const ItemTC it = locate_item(a, item, true);
  const int rows_c = chunk_rows_p(a, it.qc);
  const int U = (rows_c + 255) / 256;
  const int qcols = U * 256;
  const int k0 = it.s * a.KS2, k1 = min(it.L, k0 + a.KS2);
  const int ntiles = ceil_div_dev(k1 - k0, kPairTile);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = pair_setup(a, sm, geo, rows_c, rank);
  int issued = 0;
  if (warp == kProducerWarp) {
    if (lane == 0) issued = pair_produce<true>(a, &tq_map, &tk_map, sm, geo, it, rows_c, U, k0, ntiles, rank);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      if (rank == 0) pair_mma<true>(a, sm, geo, ntiles, U, tmem, true);
      else pair_relay(a, sm, geo, ntiles);
    }
  } else {
    if (early) pdl_wait();
    // -lse2 of every query column of the chunk (both CTAs' halves) from the
    // pass-1 partials of all key splits, stored negated; -inf marks columns
    // that do not exist.
    const int nsplit1 = ceil_div_dev(it.L, a.KS1);
    for (int row = tid; row < qcols; row += kEpiThreads)
      chunk_row_lse(a, it, row, rows_c, nsplit1, sm.nlse[row], sm.tq[row]);
    pepi_bar();
    pair_pass2_epilogue(a, sm, it, U, k0, k1, ntiles, tmem, warp, lane, rank);
  }
  pair_teardown(sm, geo, issued, tmem);
}

// ------------------------------------------------------------- host -------

template <class K>
cudaError_t launch_pair(K kernel, int pass, int items, const ScoreArgs& a, cudaStream_t s, bool pdl) {
  if (items == 0) return cudaSuccess;
  const PGeo geo = pair_geometry(pass, a.d, a.QC);
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.d, a.Hq, a.T, a.q_stride, a.q_box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.d, a.Hkv, a.T, a.k_stride, kHalf)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, geo.smem)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * items);
  cfg.blockDim = dim3(kThreadsPair);
  cfg.dynamicSmemBytes = size_t(geo.smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, mq, mk, a);
}

}  // namespace

size_t score_pair_smem_bytes(int pass, int d, int QC) { return size_t(pair_geometry(pass, d, QC).smem); }

cudaError_t launch_score_pass1_pair(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  return launch_pair(score_pass1_pair, 1, a.items1, a, s, pdl);
}

cudaError_t launch_score_pass2_pair(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  return launch_pair(score_pass2_pair, 2, a.items2, a, s, pdl);
}

}  // namespace upf
