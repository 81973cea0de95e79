// Tensor-core (tcgen05 + TMEM + TMA) scoring passes for sm_103a.
//
// UniPrefill article, section 二 first step: the last n tokens act as
// questioners and score every token; section 三: scores and their online
// normalisation are computed on the GPU.  Both passes are dense bf16
// contractions of the group's tail queries with every key, so they run on the
// 5th-generation tensor cores with fp32 accumulators in TMEM:
//
//   pass 1 (queries as M): D[q, k] = Q_rows[q, :] . K_tile[k, :]; every TMEM
//     lane is one query row, so the running (m, Z) of its causal softmax is a
//     per-thread reduction along the columns;
//   pass 2 (keys as M):    D[k, q] = K_tile[k, :] . Q_cols[q, :]; every TMEM
//     lane is one key, so sum_q 2^(x*log2e*scale - lse2[q]) is a per-thread
//     reduction along the columns.
//
// One CTA per work item (request, kv head, key split, query chunk), 18 warps:
//   warps 0-15 epilogue: warp w reads TMEM lanes 32*(w%4).. and the column
//              quarter w/4 of every unit, so all sixteen work on the same
//              unit (four warps per scheduler hide the exponential unit's and
//              the TMEM loads' latency; two were measured to leave both the
//              issue slots and the exponential unit 60% idle)
//   warp 16    TMA producer (lane 0): the query chunk once, then the key
//              tiles through a ring of 32 KB stages
//   warp 17    TMEM allocator + MMA issuer (lane 0)
// A "unit" is one MMA accumulator of 128 lanes x up to 256 fp32 columns
// (N = 256 keys per unit in pass 1, 256 query columns in pass 2; the M=128,
// N=256 shape reads 12 KB of shared memory per 128 MMA clocks, where N = 128
// would need the whole shared-memory bandwidth).  TMEM holds two such slots:
// the MMA fills one while the epilogue drains the other.  A ring stage holds
// whole key tiles (or whole 64-column slices of them), so one barrier wait and
// one tcgen05.commit cover a stage: per-slice commits were measured to stall
// the tensor pipe.
// Every wait is bounded; on a timeout the kernel records UPF_ERR_TIMEOUT, the
// roles wind down (the epilogue stops at once; a producer or MMA wait for a
// role that gave up ends on its own limit), outstanding copies and MMAs are
// waited for with the full limit, TMEM
// is freed and the kernel returns.  The pipeline waits' limit is a run-time
// argument (upf_set_wait_limit), so a test can make one expire.
#include <cuda.h>

#include <climits>
#include <cmath>

#include "score_common.cuh"
#include "sm100_ptx.cuh"
#include "upf_internal.cuh"

namespace upf {

namespace {

using namespace ptx;

constexpr int kW = 4;                          // epilogue warps per TMEM lane quarter
constexpr int kEpiWarps = 4 * kW;              // 16
constexpr int kEpiThreads = kEpiWarps * 32;    // 512
constexpr int kProducerWarp = kEpiWarps;       // 16
constexpr int kMmaWarp = kEpiWarps + 1;        // 17
constexpr int kThreadsTC = kEpiThreads + 64;   // 576
constexpr int kStageBytes = 32768;             // largest ring stage
constexpr int kMaxStages = 8;
constexpr int kMaxSlots = 4;
constexpr int kRedTiles = 8;
constexpr int kNumBars = 2 * kMaxStages + 2 * kMaxSlots + 3;   // + qfull, fin, decide                   // pass 2: tiles of per-key sums in flight
constexpr int kSmemLimit = 232448;             // opt-in dynamic shared memory per CTA
// Waits that wind a kernel down (outstanding copies and MMAs before TMEM is
// freed) always get the full limit; pipeline waits use ScoreArgs::wait_limit.
constexpr long long kWaitLimit = kDefaultWaitCycles;
constexpr uint32_t kIdleNs = 4000;              // longest suspension of a waiting role per poll

// Shape of one pass's pipeline for head dim d and QC query rows per chunk.
struct Geo {
  int S;            // 64-wide slices of the head dim (one 128-byte swizzled row each)
  int tile_keys;    // keys per tile: N of the pass-1 MMA, M (= 128) of pass 2
  int slice_bytes;  // tile_keys x 64 bf16
  int sps;          // slices per ring stage
  int spt;          // ring stages per tile
  int stage_bytes;
  int unit_cols;    // MMA N of a unit: keys (pass 1) or query columns (pass 2)
  int slot_cols;    // TMEM columns per accumulator slot
  int nslots;
  int NS;           // ring stages
  int q_bytes;      // resident query chunk: S x QC rows x 128 B
  int extra_bytes;  // pass 2: -lse2 and query positions per chunk row, per-key partial sums
  int smem;         // dynamic shared memory of the CTA
};

__host__ __device__ inline Geo geometry(int pass, int d, int QC) {
  Geo g;
  g.S = d / 64;
  g.tile_keys = (pass == 1 && d <= 128) ? 256 : 128;
  g.slice_bytes = g.tile_keys * 128;
  g.sps = imax(1, imin(g.S, kStageBytes / g.slice_bytes));
  g.spt = g.S / g.sps;
  g.stage_bytes = g.sps * g.slice_bytes;
  // Pass 2 units are 256 query columns when the chunk is a multiple of 256
  // rows, else 128; rows past the chunk's end are zero with lse2 = +inf, so
  // full-width units are exact.
  g.unit_cols = pass == 1 ? g.tile_keys : (QC % 256 == 0 ? 256 : 128);
  g.slot_cols = pass == 1 ? g.tile_keys : 256;
  g.nslots = 512 / g.slot_cols;
  g.q_bytes = g.S * QC * 128;
  g.extra_bytes = pass == 2 ? 8 * QC + kRedTiles * kW * 128 * 4 : 0;
  const int fixed = 1024 /* alignment slack */ + g.q_bytes + g.extra_bytes +
                    8 * kNumBars + 16;
  g.NS = imin(kMaxStages, (kSmemLimit - fixed) / g.stage_bytes);
  g.smem = fixed + g.NS * g.stage_bytes;
  return g;
}

// Shared-memory plan of one CTA.
struct Smem {
  unsigned char* q;       // S slices x QC rows x 128 B (1024-aligned)
  unsigned char* ring;    // NS stages
  float* nlse;            // pass 2: -lse2 per chunk row (+inf rows: -inf)
  int* tq;                // pass 2: query position per chunk row (-1: none)
  float* red;             // pass 2: [kRedTiles][kW][128] per-key sums of the column quarters
  uint64_t* bars;         // full[8], empty[8], tfull[4], tempty[4], qfull, fin, decide
  uint32_t* tmem_slot;
  int* abort_flag;
  int* redo;              // pass 1: run the item again on the checked path
};

__device__ __forceinline__ Smem carve(unsigned char* raw, const Geo& g, int QC) {
  Smem s;
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
  s.redo = reinterpret_cast<int*>(p + 12);
  return s;
}

__device__ __forceinline__ uint32_t bar_full(const Smem& sm, int st) { return smem_u32(&sm.bars[st]); }
__device__ __forceinline__ uint32_t bar_empty(const Smem& sm, int st) { return smem_u32(&sm.bars[kMaxStages + st]); }
__device__ __forceinline__ uint32_t bar_tfull(const Smem& sm, int s) { return smem_u32(&sm.bars[2 * kMaxStages + s]); }
__device__ __forceinline__ uint32_t bar_tempty(const Smem& sm, int s) {
  return smem_u32(&sm.bars[2 * kMaxStages + kMaxSlots + s]);
}
__device__ __forceinline__ uint32_t bar_qfull(const Smem& sm) {
  return smem_u32(&sm.bars[2 * kMaxStages + 2 * kMaxSlots]);
}
__device__ __forceinline__ uint32_t bar_fin(const Smem& sm) {
  return smem_u32(&sm.bars[2 * kMaxStages + 2 * kMaxSlots + 1]);
}
// Pass 1: the epilogue's verdict after the fast pass over an item (one arrival).
__device__ __forceinline__ uint32_t bar_decide(const Smem& sm) {
  return smem_u32(&sm.bars[2 * kMaxStages + 2 * kMaxSlots + 2]);
}

__device__ __forceinline__ void init_barriers(const Smem& sm) {
  for (int i = 0; i < kMaxStages; ++i) {
    mbar_init(bar_full(sm, i), 1);
    mbar_init(bar_empty(sm, i), 1);
  }
  for (int s = 0; s < kMaxSlots; ++s) {
    mbar_init(bar_tfull(sm, s), 1);
    mbar_init(bar_tempty(sm, s), kEpiWarps);   // every epilogue warp drains every unit
  }
  mbar_init(bar_qfull(sm), 1);
  mbar_init(bar_fin(sm), 1);
  mbar_init(bar_decide(sm), 1);
  *sm.abort_flag = 0;
  *sm.redo = 0;
  fence_barrier_init();
}

__device__ __forceinline__ bool aborted(const Smem& sm) { return *reinterpret_cast<volatile int*>(sm.abort_flag) != 0; }

__device__ __forceinline__ void abort_with_timeout(const ScoreArgs& a, const Smem& sm) {
  set_status(a.status, UPF_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
}

// Rows of the query chunk present in this item: [0, rows_c).
__device__ __forceinline__ int chunk_rows(const ScoreArgs& a, int qc) { return min(a.QC, a.QR - qc * a.QC); }

// Zero the rows [rows_c, pad) of the query chunk (generic stores, ordered
// before any MMA reads by the caller's proxy fence + barrier).
__device__ __forceinline__ void zero_padding(const ScoreArgs& a, const Smem& sm, int rows_c, int pad) {
  const int n16 = (pad - rows_c) * 8;
  for (int s = 0; s < a.d / 64; ++s) {
    uint4* base = reinterpret_cast<uint4*>(sm.q + size_t(s) * a.QC * 128 + size_t(rows_c) * 128);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
  }
}

// An epilogue warp is done reading a TMEM slot: order its loads before the
// arrival the MMA issuer waits for.
__device__ __forceinline__ void release_slot(const Smem& sm, int slot, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_tempty(sm, slot));
}

// Wait until the MMA has filled `slot` for the use with phase parity `parity`;
// false (and the abort flag set) on a timeout or another role's abort.
__device__ __forceinline__ bool wait_slot(const ScoreArgs& a, const Smem& sm, int slot, uint32_t parity) {
  if (aborted(sm)) return false;
  if (!mbar_wait_idle(bar_tfull(sm, slot), parity, a.wait_limit, kIdleNs)) {
    abort_with_timeout(a, sm);
    return false;
  }
  tc_fence_after();
  return true;
}

// wait_slot with the common case first: the unit is already there.
__device__ __forceinline__ bool wait_slot_fast(const ScoreArgs& a, const Smem& sm, int slot, uint32_t parity) {
  if (mbar_try_wait(bar_tfull(sm, slot), parity)) {
    tc_fence_after();
    return true;
  }
  return wait_slot(a, sm, slot, parity);
}

// --------------------------------------------------- producer and MMA -----

// Producer: the query chunk (once), then every key tile stage by stage
// (pass 1: a second time when the epilogue's verdict asks for it).  Returns
// the number of stage loads issued.  Called by one lane, or (warp_wide) by the
// whole warp, which runs the bookkeeping and the waits with warp-uniform values
// while one elected lane issues the copies.
__device__ int produce(const ScoreArgs& a, const CUtensorMap* tq_map, const CUtensorMap* tk_map, const Smem& sm,
                       const Geo& geo, const ItemTC& it, int rows_c, int k0, int ntiles, bool may_repeat,
                       bool warp_wide, bool descending = false) {
  const bool leader = warp_wide ? elect_one() : true;
  const int BQ = a.q_box_rows;
  const int boxes = rows_c / BQ;
  if (leader) mbar_arrive_expect_tx(bar_qfull(sm), uint32_t(boxes) * geo.S * BQ * 128);
  for (int b = 0; b < boxes; ++b) {
    const int rho = it.qc * a.QC + b * BQ;
    const int h = a.qhead[it.g * a.gamma + rho / a.n];
    const int tok = it.tok0 + it.L - a.n + rho % a.n;   // may be < 0 or in another request; masked later
    if (leader)
      for (int s = 0; s < geo.S; ++s)
        tma_load_3d(smem_u32(sm.q + size_t(s) * a.QC * 128 + size_t(b) * BQ * 128), tq_map, s * 64, h, tok,
                    bar_qfull(sm));
  }
  const int total = ntiles * geo.spt;
  int q = 0, st = 0;
  uint32_t ph = 0;
  for (int round = 0; round < (may_repeat ? 2 : 1); ++round) {
    if (round == 1) {   // pass 1: the tiles again only if the epilogue asks for it
      if (!mbar_wait_idle(bar_decide(sm), 0, a.wait_limit, kIdleNs)) {
        abort_with_timeout(a, sm);
        break;
      }
      if (*reinterpret_cast<volatile int*>(sm.redo) == 0) break;
    }
    const int step = descending ? -geo.tile_keys : geo.tile_keys;
    int part = 0, key = it.tok0 + k0 + (descending ? (ntiles - 1) * geo.tile_keys : 0);
    for (int n = 0; n < total; ++n, ++q) {
      if (!mbar_wait_idle(bar_empty(sm, st), ph ^ 1u, a.wait_limit, kIdleNs)) {
        abort_with_timeout(a, sm);
        return q;
      }
      const uint32_t dst = smem_u32(sm.ring) + uint32_t(st * geo.stage_bytes);
      if (leader) {
        mbar_arrive_expect_tx(bar_full(sm, st), uint32_t(geo.stage_bytes));
        for (int ss = 0; ss < geo.sps; ++ss)
          tma_load_3d(dst + uint32_t(ss * geo.slice_bytes), tk_map, (part * geo.sps + ss) * 64, it.g, key,
                      bar_full(sm, st));
      }
      if (++st == geo.NS) { st = 0; ph ^= 1u; }
      if (++part == geo.spt) { part = 0; key += step; }
    }
  }
  return q;
}

// After an abort: wait (bounded) for the query load and for the last key
// load issued into each stage, so no copy is still landing when the CTA exits.
__device__ void drain_loads(const Smem& sm, const Geo& geo, int issued) {
  mbar_wait(bar_qfull(sm), 0, kWaitLimit / 8);
  for (int st = 0; st < geo.NS; ++st) {
    const int c = issued > st ? (issued - st + geo.NS - 1) / geo.NS : 0;   // loads issued into stage st
    if (c > 0) mbar_wait(bar_full(sm, st), (c - 1) & 1, kWaitLimit / 8);
  }
}

// One thread issues every unit's MMAs in order.  Pass 1 (keys_as_m false):
// unit u of a tile is query rows [128u, 128u+128) (A) against the tile's
// tile_keys keys (B, N = tile_keys).  Pass 2: the tile's 128 keys (A) against
// query columns [W u, W u + W) (B, N = W = unit_cols).  Before returning it waits for all of
// them to finish.  Called by one lane, or (warp_wide) by the whole warp, which
// runs the loop with warp-uniform descriptors and counters while the elected
// lane issues every MMA and commit (a commit tracks the MMAs of the thread
// that issues it).  Measured on the 128K-token LLaMA shape, the warp-wide
// form makes pass 1 about 3 % faster and pass 2 about 3 % slower, so pass 2
// keeps one lane.
template <bool kEarly>
__device__ void issue_mma(const ScoreArgs& a, const Smem& sm, const Geo& geo, int ntiles, int units, uint32_t tmem,
                          bool keys_as_m, bool may_repeat, bool warp_wide) {
  const bool leader = warp_wide ? elect_one() : true;
  // Division-free bookkeeping: this thread shares its scheduler with busy
  // epilogue warps, so every instruction between two MMAs costs issue slots.
  const uint32_t idesc = idesc_bf16_f32(128, uint32_t(geo.unit_cols));
  const uint32_t ring0 = smem_u32(sm.ring), q0 = smem_u32(sm.q);
  const uint32_t q_slice = uint32_t(a.QC) * 128u;
  const uint32_t q_unit = uint32_t(keys_as_m ? geo.unit_cols : 128) * 128u;
  bool ok = mbar_wait_idle(bar_qfull(sm), 0, a.wait_limit, kIdleNs);
  int st = 0;            // ring stage of the next tile's first part
  uint32_t ph = 0;       // its phase parity
  int slot = 0;          // TMEM slot of the next unit
  uint32_t sph = 0;      // its phase parity
  for (int round = 0; ok && round < (may_repeat ? 2 : 1); ++round) {
  if (round == 1) {        // pass 1: the tiles again only if the epilogue asks for it
    ok = mbar_wait_idle(bar_decide(sm), 0, a.wait_limit, kIdleNs);
    if (!ok || *reinterpret_cast<volatile int*>(sm.redo) == 0) break;
  }
  for (int i = 0; ok && i < ntiles; ++i) {
    // A tile takes spt <= 2 consecutive ring stages; slice s lives in stage
    // part s / sps at offset (s % sps) slices, sps in {1, 2}.
    // No abort test in this loop: every extra instruction of the issuing
    // thread, which shares its scheduler with busy epilogue warps, was measured
    // to cost 2-3 % of the pass; once another role gave up, these waits end on
    // their own limit.
    // With two stages per tile (kEarly), the tile's first unit starts on the
    // first stage while the second may still be landing, and the first stage
    // is released as soon as the last unit has read it: the next tile's second
    // load then has about two units of MMA work to arrive behind, not none.
    // Measured faster in pass 1 and in pass 2 with two or more units per tile;
    // with one unit per tile the pass-2 release is a commit in the middle of a
    // unit, which stalls the tensor pipe more than the earlier load gains.  A
    // compile-time choice: even the untaken tests cost this thread's loop time.
    const int st0 = st, st1 = st + 1 == geo.NS ? 0 : st + 1;
    const uint32_t ph1 = st1 == 0 ? ph ^ 1u : ph;
    const bool two = kEarly && geo.spt == 2;
    ok = mbar_wait_idle(bar_full(sm, st0), ph, a.wait_limit, kIdleNs);
    if (!kEarly && ok && geo.spt == 2) ok = mbar_wait_idle(bar_full(sm, st1), ph1, a.wait_limit, kIdleNs);
    if (geo.spt == 2) { st = st1 + 1 == geo.NS ? 0 : st1 + 1; ph = (st1 == 0 || st == 0) ? ph ^ 1u : ph; }
    else { st = st1; ph = st1 == 0 ? ph ^ 1u : ph; }
    const uint32_t k0a = ring0 + uint32_t(st0 * geo.stage_bytes), k1a = ring0 + uint32_t(st1 * geo.stage_bytes);
    if (!ok) break;
    tc_fence_after();
    for (int u = 0; u < units; ++u) {
      ok = mbar_wait_idle(bar_tempty(sm, slot), sph ^ 1u, a.wait_limit, kIdleNs);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dt = tmem + uint32_t(slot * geo.slot_cols);
      const uint32_t qu = q0 + uint32_t(u) * q_unit;
      for (int s = 0; s < geo.S; ++s) {
        if (kEarly && two && s == geo.sps) {   // the first slice of the second stage
          if (u == units - 1 && leader) mma_commit(bar_empty(sm, st0));
          if (u == 0) {
            ok = mbar_wait_idle(bar_full(sm, st1), ph1, a.wait_limit, kIdleNs);
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
          if (leader) mma_bf16(dt, da + uint64_t(2 * kk), db + uint64_t(2 * kk), idesc, (s | kk) ? 1u : 0u);
      }
      if (kEarly && !ok) break;
      if (leader) mma_commit(bar_tfull(sm, slot));
      if (++slot == geo.nslots) { slot = 0; sph ^= 1u; }
    }
    if (!ok) break;
    if (leader) {
      if (!kEarly) {
        mma_commit(bar_empty(sm, st0));
        if (geo.spt == 2) mma_commit(bar_empty(sm, st1));
      } else {
        mma_commit(bar_empty(sm, two ? st1 : st0));
      }
    }
  }
  }
  if (!ok) abort_with_timeout(a, sm);
  // Every MMA this warp issued must be done before TMEM can be freed: this
  // wait keeps the full limit whatever the pipeline limit is.  If even it
  // expires, the error is recorded and TMEM is still freed (a CTA that left
  // its columns allocated would stall the next CTA's allocation on this SM).
  if (leader) mma_commit(bar_fin(sm));
  if (!mbar_wait_idle(bar_fin(sm), 0, kWaitLimit, kIdleNs)) abort_with_timeout(a, sm);
}

// Common prologue of both passes: barriers, padding, TMEM; returns the TMEM base.
__device__ __forceinline__ uint32_t setup(const ScoreArgs& a, const Smem& sm, int rows_c, int pad) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) init_barriers(sm);
  zero_padding(a, sm, rows_c, pad);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(sm.tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *sm.tmem_slot;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

// Pass 2: the kW column-quarter sums of key row `krow` of tile i, in order.
__device__ __forceinline__ float red_sum(const float* red, int i, int krow) {
  const float* r = red + (i % kRedTiles) * kW * 128 + krow;
  float t = r[0];
#pragma unroll
  for (int c = 1; c < kW; ++c) t += r[c * 128];
  return t;
}



// ------------------------------------------------------------- pass 1 -----

template <bool B>
struct Flag {
  static constexpr bool value = B;
};

// OR of a predicate over the epilogue warps (named barrier 1 with reduction).
__device__ __forceinline__ int epi_bar_or(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.s32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(kEpiThreads)
      : "memory");
  return r;
}

// Epilogue of pass 1.  This thread is row 128h + 32qd + lane of every unit h
// and covers the column quarter cb of it (CPW chunks of 32 keys); it keeps
// (m, Z) of up to four rows in registers.  At the end the quarters of every
// row are merged through shared memory and one (m, Z) per row is stored.
//
// An item is swept once on a fast path: the first key tile sets every row's
// reference m to its maximum, later tiles add their exponential sums with no
// test in the way (a test per unit made each unit's sums stall the warp) and
// only note, in a flag, a sum that is not finite (a logit more than about 127
// above the first tile's maximum).  Rows whose m is still -inf after the first
// tile see no key of the item at all (keys are visible up to a position, and
// the first tile holds the item's lowest keys) and are skipped.  If any row of
// the CTA was flagged, the epilogue says so through the decide barrier and
// the producer, the MMA and the epilogue sweep the item again on the checked
// path, which moves m whenever a unit's sums leave [0, 2^20].
template <int CPW>
__device__ __forceinline__ void pass1_epilogue(const ScoreArgs& a, const Smem& sm, const Geo& geo, const ItemTC& it,
                                               int item, int rows_c, int MT, int k0, int ntiles, uint32_t tmem,
                                               int warp, int lane) {
  const int qd = warp & 3, cb = warp >> 2;
  const int span = CPW * 32;   // = tile_keys / kW
  const float sl = a.scale_log2;
  const int r0 = qd * 32 + lane;
  // Per row: the last key this warp's columns may see, relative to the
  // tile's first key (INT_MIN: not a row of the chunk).
  auto lim_of = [&](int h) {
    const int row = h * 128 + r0;
    return (h < MT && row < rows_c) ? it.L - a.n + (it.qc * a.QC + row) % a.n - cb * span : INT_MIN;
  };
  const int l0 = lim_of(0), l1 = lim_of(1), l2 = lim_of(2), l3 = lim_of(3);
  float m0, m1, m2, m3, z0, z1, z2, z3;
  const uint32_t tbase = tmem + (uint32_t(qd * 32) << 16) + uint32_t(cb * span);
  bool ok = true;
  // TMEM slot of the next unit and its phase parity, advanced without a
  // division (the slot count is 2 or 4, known only at run time); the sequence
  // continues into a second sweep as the MMA's does.
  int slot_next = 0;
  uint32_t slot_par = 0;
  auto sweep = [&](auto checked_flag) -> bool {   // returns: some sum not finite (fast path only)
    constexpr bool kChecked = decltype(checked_flag)::value;
    m0 = m1 = m2 = m3 = -INFINITY;
    z0 = z1 = z2 = z3 = 0.f;
    bool bad = false;
    for (int i = 0; ok && i < ntiles; ++i) {
      const int kt = k0 + i * geo.tile_keys;   // request-relative first key of the tile
      const bool masked = kt + geo.tile_keys - 1 > it.L - a.n;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (h >= MT) break;
        const int slot = slot_next;
        if (!wait_slot_fast(a, sm, slot, slot_par)) {
          ok = false;
          break;
        }
        if (++slot_next == geo.nslots) {
          slot_next = 0;
          slot_par ^= 1u;
        }
        const int lh = h == 0 ? l0 : h == 1 ? l1 : h == 2 ? l2 : l3;
        float mh = h == 0 ? m0 : h == 1 ? m1 : h == 2 ? m2 : m3;
        float zh = h == 0 ? z0 : h == 1 ? z1 : h == 2 ? z2 : z3;
        const bool live = lh != INT_MIN;
        const int lim = live ? lh - kt : 0;   // this warp's columns j > lim are invisible
        // Both chunks are loaded before one wait and the slot is released
        // before the math.
        float va[32], vb[32];
        const uint32_t ta = tbase + uint32_t(slot * geo.slot_cols);
        tmem_ld32(ta, va);
        if (CPW == 2) tmem_ld32(ta + 32u, vb);
        tmem_wait_ld();
        release_slot(sm, slot, lane);
        if (masked) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j > lim) va[j] = -INFINITY;
            if (CPW == 2 && 32 + j > lim) vb[j] = -INFINITY;
          }
        }
        if (live) {
          if (kChecked) {
            const float sa = exp_sum32(va, sl, mh);
            const float sb = CPW == 2 ? exp_sum32(vb, sl, mh) : 0.f;
            if (sa <= 1048576.f && sb <= 1048576.f) zh += sa + sb;
            else online_rescale<CPW>(va, vb, sl, mh, zh);
          } else if (i == 0) {
            online_rescale<CPW>(va, vb, sl, mh, zh);   // the reference: the first tile's maximum
          } else if (mh > -INFINITY) {
            const float t = exp_sum32(va, sl, mh) + (CPW == 2 ? exp_sum32(vb, sl, mh) : 0.f);
            zh += t;
            bad |= !(t <= 3.0e38f);
          }
        }
        if (h == 0) { m0 = mh; z0 = zh; }
        else if (h == 1) { m1 = mh; z1 = zh; }
        else if (h == 2) { m2 = mh; z2 = zh; }
        else { m3 = mh; z3 = zh; }
      }
    }
    return bad || !(z0 <= 3.0e38f && z1 <= 3.0e38f && z2 <= 3.0e38f && z3 <= 3.0e38f);
  };
  const bool bad = sweep(Flag<false>{}) && ok;
  const int redo = epi_bar_or(bad ? 1 : 0) && !aborted(sm);
  if (threadIdx.x == 0) {
    *reinterpret_cast<volatile int*>(sm.redo) = redo;
    mbar_arrive(bar_decide(sm));
  }
  if (redo) sweep(Flag<true>{});
  // The ring is idle here: every MMA, hence every load, finished before the
  // last unit was read, and no second sweep follows.
  float2* red = reinterpret_cast<float2*>(sm.ring);   // [kW][QC]
  if (ok) {
    red[cb * a.QC + r0] = make_float2(m0, z0);
    if (MT > 1) red[cb * a.QC + 128 + r0] = make_float2(m1, z1);
    if (MT > 2) red[cb * a.QC + 256 + r0] = make_float2(m2, z2);
    if (MT > 3) red[cb * a.QC + 384 + r0] = make_float2(m3, z3);
  }
  epi_bar();
  if (!ok || aborted(sm)) return;
  for (int row = cb * 128 + r0; row < MT * 128; row += kW * 128) {
    if (row >= rows_c) continue;
    float mm = -INFINITY;
#pragma unroll
    for (int c = 0; c < kW; ++c) mm = fmaxf(mm, red[c * a.QC + row].x);
    float zz = 0.f;
    if (mm > -INFINITY) {
#pragma unroll
      for (int c = 0; c < kW; ++c) {
        const float2 p = red[c * a.QC + row];
        if (p.y > 0.f) zz += p.y * ex2_approx(p.x - mm);
      }
    }
    a.p1part[(int64_t)item * a.QC + row] = make_float2(mm, zz);
  }
}

__global__ void __launch_bounds__(kThreadsTC, 1)
    score_pass1_tc(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                   const __grid_constant__ ScoreArgs a) {
  // Wait, then let pass 2 launch: pass 2 may read the queries and keys before
  // its own wait, so it must not start before this kernel's predecessor (which
  // may have written them) is complete.
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x;
  if (!item_exists(a, item, false)) return;
  const Geo geo = geometry(1, a.d, a.QC);
  const Smem sm = carve(smem_raw, geo, a.QC);
  const ItemTC it = locate_item(a, item, false);
  const int rows_c = chunk_rows(a, it.qc);
  const int k0 = it.s * a.KS1, k1 = min(it.L, k0 + a.KS1);
  const int ntiles = ceil_div_dev(k1 - k0, geo.tile_keys);
  const int MT = (rows_c + 127) / 128;   // units per tile: 128-row blocks of the chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = setup(a, sm, rows_c, MT * 128);

  int issued = 0;
  if (warp == kProducerWarp) {
    issued = produce(a, &tq_map, &tk_map, sm, geo, it, rows_c, k0, ntiles, true, true);
    if (blockIdx.x == 0) desc_check(a, lane);
  } else if (warp == kMmaWarp) {
    issue_mma<true>(a, sm, geo, ntiles, MT, tmem, false, true, true);
  } else if (geo.tile_keys / kW == 64) {
    pass1_epilogue<2>(a, sm, geo, it, item, rows_c, MT, k0, ntiles, tmem, warp, lane);
  } else {
    pass1_epilogue<1>(a, sm, geo, it, item, rows_c, MT, k0, ntiles, tmem, warp, lane);
  }
  // Wind down: outstanding loads of an aborted pipeline, then free TMEM.
  if (warp == kProducerWarp && lane == 0 && aborted(sm)) drain_loads(sm, geo, issued);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------- pass 2 -----

// Epilogue of pass 2.  This thread is key 32qd + lane of every tile; its warp
// reads the 32-column chunks cb and cb + kW (CPW of them) of every unit and
// stores its per-key sum in red[i % kRedTiles][cb] without waiting.  A warp
// holding unit x knows every warp released unit x - 2 (the MMA reuses a slot
// only after that), so every warp finished all tiles before the one holding
// unit x - 2, stores included (mbarrier arrive/wait order them): with two or
// more units per tile, tile i - 2 is complete once a warp holds tile i, with
// one unit tile i - 3 (the lag D).  The quarter's first warp adds the kW sums
// of tile i - D in a fixed order (so results are reproducible) and writes
// them out at the start of tile i; a row is rewritten D tiles after that read
// is known done (kRedTiles >= 2D); the last D tiles go out after a barrier.
template <int CPW>
__device__ __forceinline__ void pass2_epilogue(const ScoreArgs& a, const Smem& sm, const Geo& geo, const ItemTC& it,
                                               int U, int k0, int k1, int ntiles, uint32_t tmem, int warp,
                                               int lane) {
  const int qd = warp & 3, cb = warp >> 2;
  const int krow = qd * 32 + lane;
  const float sl = a.scale_log2;
  float* out = a.part + (int64_t)(it.g * a.NQC + it.qc) * a.T + it.tok0;
  const uint32_t tq = tmem + (uint32_t(qd * 32) << 16) + uint32_t(cb * 32);
  const int lag = U >= 2 ? 2 : 3;
  const uint32_t nlse_s = smem_u32(sm.nlse);
  static_assert(kRedTiles >= 6, "rows are read lag tiles after their stores and rewritten lag tiles later");
  bool ok = true;
  int uidx = 0;
  // Tiles run from the item's last keys to its first: pass 1 read the keys in
  // ascending order, so the last ones it read may still be in L2.
  for (int i = 0; i < ntiles; ++i) {
    const int kt = k0 + (ntiles - 1 - i) * geo.tile_keys;
    const int key = kt + krow;
    const bool masked = kt + geo.tile_keys - 1 > it.L - a.n;
    uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);
    for (int u = 0; u < U; ++u, ++uidx) {
      const int slot = uidx & 1;
      if (!wait_slot_fast(a, sm, slot, (uidx >> 1) & 1)) {
        ok = false;
        break;
      }
      if (u == 0 && cb == 0 && i >= lag) {   // tile i - lag is complete: write it out
        const int kprev = key + lag * geo.tile_keys;
        if (kprev < k1) out[kprev] = red_sum(sm.red, i - lag, krow);
      }
      const int col0 = u * geo.unit_cols + cb * 32;
      {   // both chunks loaded, one wait, the slot released, then the math
        float va[32], vb[32];
        const uint32_t ta = tq + uint32_t(slot * 256);
        tmem_ld32(ta, va);
        if (CPW == 2) tmem_ld32(ta + uint32_t(32 * kW), vb);
        tmem_wait_ld();
        release_slot(sm, slot, lane);
        if (!masked) {
          normalised_sum32(va, nlse_s + 4 * col0, sl, acc0, acc1);
          if (CPW == 2) normalised_sum32(vb, nlse_s + 4 * (col0 + 32 * kW), sl, acc0, acc1);
        } else {
          float t = normalised_sum32_masked(va, sm.nlse + col0, sm.tq + col0, key, sl);
          if (CPW == 2) t += normalised_sum32_masked(vb, sm.nlse + col0 + 32 * kW, sm.tq + col0 + 32 * kW, key, sl);
          acc0 = add2(acc0, pack2(t, 0.f));
        }
      }
    }
    if (!ok) break;
    float lo, hi;
    unpack2(add2(acc0, acc1), lo, hi);
    sm.red[((i % kRedTiles) * kW + cb) * 128 + krow] = lo + hi;
  }
  epi_bar();
  if (ok && cb == 0 && !aborted(sm))
    for (int i = max(0, ntiles - lag); i < ntiles; ++i) {
      const int key = k0 + (ntiles - 1 - i) * geo.tile_keys + krow;
      if (key < k1) out[key] = red_sum(sm.red, i, krow);
    }
}

__global__ void __launch_bounds__(kThreadsTC, 1)
    score_pass2_tc(const __grid_constant__ CUtensorMap tq_map, const __grid_constant__ CUtensorMap tk_map,
                   const __grid_constant__ ScoreArgs a) {
  // With the descriptor in the parameters, nothing before the -lse merge reads
  // what pass 1 writes: the set-up, the query and key loads and the first
  // MMAs run while pass 1's last CTAs finish, and only the epilogue waits for
  // pass 1 (which launched this kernel after its own predecessor completed).
  // Tables in the workspace come from the describe kernel, so then every
  // thread waits first.
  const bool early = a.desc.R > 0;
  pdl_trigger();
  if (!early) pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  const int item = blockIdx.x;
  if (!item_exists(a, item, true)) return;
  const Geo geo = geometry(2, a.d, a.QC);
  const Smem sm = carve(smem_raw, geo, a.QC);
  const ItemTC it = locate_item(a, item, true);
  const int rows_c = chunk_rows(a, it.qc);
  const int U = (rows_c + geo.unit_cols - 1) / geo.unit_cols;   // units per tile
  const int qcols = U * geo.unit_cols;                         // MMA columns (zero-padded query rows)
  const int k0 = it.s * a.KS2, k1 = min(it.L, k0 + a.KS2);
  const int ntiles = ceil_div_dev(k1 - k0, geo.tile_keys);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = setup(a, sm, rows_c, qcols);

  int issued = 0;
  if (warp == kProducerWarp) {
    if (lane == 0) issued = produce(a, &tq_map, &tk_map, sm, geo, it, rows_c, k0, ntiles, false, false, true);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      if (U >= 2) issue_mma<true>(a, sm, geo, ntiles, U, tmem, true, false, false);
      else issue_mma<false>(a, sm, geo, ntiles, U, tmem, true, false, false);
    }
  } else {
    // lse2 of every query row of the chunk from the pass-1 partials (all key
    // splits), stored negated; -inf marks rows that do not exist (padding,
    // or positions before the request start).  The MMA runs meanwhile: the
    // first unit is not read before this is done.  The parameter reads come
    // before the wait (a chunk has at most kEpiThreads rows).
    const int nsplit1 = ceil_div_dev(it.L, a.KS1);
    const int64_t split_stride = (int64_t)a.NQC1 * a.QC1;   // consecutive pass-1 splits of one (g, qc)
    const LseRow mine = tid < qcols ? lse_row_prep(a, it, tid, rows_c, nsplit1) : LseRow{nullptr, -1};
    if (early) pdl_wait();
    if (tid < qcols) lse_row_finish(mine, nsplit1, split_stride, sm.nlse[tid], sm.tq[tid]);
    for (int row = tid + kEpiThreads; row < qcols; row += kEpiThreads)
      chunk_row_lse(a, it, row, rows_c, nsplit1, sm.nlse[row], sm.tq[row]);
    epi_bar();
    if (geo.unit_cols == 256) pass2_epilogue<2>(a, sm, geo, it, U, k0, k1, ntiles, tmem, warp, lane);
    else pass2_epilogue<1>(a, sm, geo, it, U, k0, k1, ntiles, tmem, warp, lane);
  }
  if (warp == kProducerWarp && lane == 0 && aborted(sm)) drain_loads(sm, geo, issued);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------- host -------

static_assert(sizeof(ScoreArgs) + 2 * sizeof(CUtensorMap) <= 4096, "scoring kernel parameters within 4 KB");

template <class K>
cudaError_t launch_pass(K kernel, int pass, int items, const ScoreArgs& a, cudaStream_t s, bool pdl) {
  if (items == 0) return cudaSuccess;
  const Geo geo = geometry(pass, a.d, a.QC);
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.d, a.Hq, a.T, a.q_stride, a.q_box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.d, a.Hkv, a.T, a.k_stride, geo.tile_keys)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, geo.smem)) != cudaSuccess)
    return e;
  return launch_kernel(kernel, items, kThreadsTC, size_t(geo.smem), s, pdl, mq, mk, a);
}

}  // namespace

int score_tc_key_tile(int pass, int d) { return geometry(pass, d, 128).tile_keys; }
size_t score_tc_smem_bytes(int pass, int d, int QC) { return size_t(geometry(pass, d, QC).smem); }

cudaError_t launch_score_pass1_tc(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  return launch_pass(score_pass1_tc, 1, a.items1, a, s, pdl);
}

cudaError_t launch_score_pass2_tc(const ScoreArgs& a, cudaStream_t s, bool pdl) {
  return launch_pass(score_pass2_tc, 2, a.items2, a, s, pdl);
}

}  // namespace upf
