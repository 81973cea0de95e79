// The per-request top-p block selection shared by the selection kernels.
//
// UniPrefill article, section 二 second step: rank the blocks by their mean
// token importance and keep the smallest set whose importance sum reaches p
// of the total; exemption paragraph: blocks covering the first and last 128
// tokens are always kept.
//
// One CTA (kSelThreads threads) selects one request's blocks.  Block masses
// become 48-bit fixed-point integers relative to the request's largest block,
// so totals and histograms are exact integer sums (deterministic in any
// order; rounding below 1e-10 of the total).  Non-negative float bit patterns
// order like the values, so an MSB-first radix select over the 32-bit
// patterns (8 bits per round, integer mass and count histograms in shared
// memory) narrows down the bucket holding the boundary: the block whose mass
// brings the ranked prefix (score desc, index asc) to p of the total.  Blocks
// above the bucket are in.  Once the bucket holds at most kCountSel blocks
// (usually after the first round) its blocks are listed and each is kept when
// the mass ranked before it is below the target, counted by one thread per
// candidate; a bucket that never gets that small (many equal scores) ends
// after four rounds with one score v*, whose blocks enter in index order
// until the mass is reached.  No sort.
//
// Histogram updates are aggregated per warp before the shared-memory atomics:
// the blocks of a request have similar magnitudes, so in the first rounds most
// of them share a few digits, and one atomic per block would serialise on
// those few addresses.  Lanes with the digit of the lowest pending lane add
// their masses with full-warp reductions of the masses' 16-bit parts, and one
// lane adds the group's sums and count.
#pragma once

#include <cmath>

#include "upf_internal.cuh"

namespace upf {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kCountSel = 256;   // requests (and boundary buckets) of up to this many blocks are ranked by counting

// Shared memory the select core needs beyond its static arrays, for a request
// of up to nbp blocks (nbp a multiple of 8).
__host__ __device__ constexpr size_t select_smem_bytes(int nbp) {
  return size_t(nbp) * (sizeof(unsigned long long) + sizeof(uint32_t) + 1);
}

struct SelectScratch {
  unsigned long long* m;   // [nbp] fixed-point masses
  uint32_t* bits;          // [nbp] float bits of the block scores
  unsigned char* keep;     // [nbp] 1 = kept
};

__device__ __forceinline__ SelectScratch carve_select(unsigned char* dyn, int nbp) {
  SelectScratch s;
  s.m = reinterpret_cast<unsigned long long*>(dyn);
  s.bits = reinterpret_cast<uint32_t*>(s.m + nbp);
  s.keep = reinterpret_cast<unsigned char*>(s.bits + nbp);
  return s;
}

// Block masses as 48-bit fixed point relative to the largest block of the
// request: m = floor(v * 2^sh), sh = 48 - ex with vmax = f * 2^ex, f in
// [0.5, 1), so every m < 2^48 and a request's total (<= 16384 blocks) stays
// below 2^62.  Exact, from the float's fields: v (>= 0, <= vmax) is
// mant * 2^(e - 150) with e the biased exponent (1 for subnormals), so m is
// mant shifted by e - 150 + sh (at most 25 to the left).
__device__ __forceinline__ unsigned long long fixed_mass(float v, int sh) {
  const uint32_t b = __float_as_uint(v);
  const int e = int(b >> 23);
  const uint32_t mant = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  const int s = (e ? e : 1) - 150 + sh;
  if (s >= 0) return (unsigned long long)mant << s;
  return s > -32 ? (unsigned long long)(mant >> -s) : 0ull;
}

// The smallest integer >= top_p * total, exactly, for top_p in [0, 1] and
// total < 2^62: top_p = mp / 2^k with mp the 24-bit significand, so the
// answer is the 88-bit product mp * total shifted right by k, rounded up.
// Integer arithmetic throughout (no double precision, which is slow here).
__device__ __forceinline__ unsigned long long mass_target(float top_p, unsigned long long total) {
  const uint32_t b = __float_as_uint(top_p);
  const int e = int(b >> 23) & 0xFF;
  const unsigned long long mp = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  const int k = 150 - (e ? e : 1);   // >= 23 for top_p <= 1
  const unsigned long long lo = total * mp, hi = __umul64hi(total, mp);
  unsigned long long q;
  bool rem;
  if (k < 64) {
    q = (hi << (64 - k)) | (lo >> k);
    rem = (lo & ((1ull << k) - 1ull)) != 0;
  } else if (k < 128) {
    q = k == 64 ? hi : hi >> (k - 64);
    rem = lo != 0 || (k > 64 && (hi & ((1ull << (k - 64)) - 1ull)) != 0);
  } else {
    q = 0;
    rem = lo != 0 || hi != 0;
  }
  return q + (rem ? 1ull : 0ull);
}

// Cross-warp reductions of one value per warp (kSelWarps == 32: lane w reads
// warp w's value), each one warp instruction in every warp, so no thread
// walks the array.  Integer sums, maxima and ORs do not depend on the order.
static_assert(kSelWarps == 32, "one per-warp value per lane");

// Sum over the warp's lanes of v (each < 2^62, the sum < 2^64) in three
// 21-bit parts, so no 32-bit part sum overflows.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
  const uint32_t p0 = __reduce_add_sync(0xffffffffu, uint32_t(v & 0x1FFFFFull));
  const uint32_t p1 = __reduce_add_sync(0xffffffffu, uint32_t((v >> 21) & 0x1FFFFFull));
  const uint32_t p2 = __reduce_add_sync(0xffffffffu, uint32_t(v >> 42));
  return (unsigned long long)p0 + ((unsigned long long)p1 << 21) + ((unsigned long long)p2 << 42);
}

// Sum of the values of the warps before this one.
__device__ __forceinline__ int warps_before_sum(const int* s_w) {
  const int lane = threadIdx.x & 31;
  return __reduce_add_sync(0xffffffffu, lane < (int(threadIdx.x) >> 5) ? s_w[lane] : 0);
}

// The CTA's sum of v (the total < 2^62); every thread gets it.
__device__ __forceinline__ unsigned long long sel_block_sum(unsigned long long v, unsigned long long* s_tmp) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) s_tmp[threadIdx.x >> 5] = v;
  __syncthreads();
  return warp_sum_u64(s_tmp[threadIdx.x & 31]);   // s_tmp is written again only after later barriers
}

// Mass histograms are kept as three 32-bit histograms of the masses' 16-bit
// parts (native 32-bit shared atomics; a bucket's part sum stays below
// 16384 * 2^16 = 2^30), combined when the buckets are scanned, beside the
// buckets' block counts.
struct MassHist {
  uint32_t p[3][256];
  uint32_t c[256];
};
constexpr int kHistWords = 4 * 256;

__device__ __forceinline__ unsigned long long hist_mass(const MassHist& h, int d) {
  return (unsigned long long)h.p[0][d] + ((unsigned long long)h.p[1][d] << 16) + ((unsigned long long)h.p[2][d] << 32);
}

// Adds `mass` to bucket `digit` for every lane with digit < 256.  Every lane
// of the warp calls it (lanes with nothing to add pass digit >= 256).  Up to
// four times, the lanes sharing the digit of the lowest lane still pending add
// their masses with full-warp reductions of the 16-bit parts (no sum overflows
// 32 bits) and one lane does the shared atomics; lanes left after that (digits
// already spread out) add their own.
__device__ __forceinline__ void hist_add_aggregated(MassHist& h, uint32_t digit, unsigned long long mass) {
  const int lane = threadIdx.x & 31;
  const uint32_t m0 = uint32_t(mass & 0xFFFFull), m1 = uint32_t((mass >> 16) & 0xFFFFull), m2 = uint32_t(mass >> 32);
  unsigned pending = __ballot_sync(0xffffffffu, digit < 256u);
#pragma unroll 1
  for (int it = 0; it < 4 && pending; ++it) {
    const int leader = __ffs(pending) - 1;
    const uint32_t d = __shfl_sync(0xffffffffu, digit, leader);
    const bool mine = ((pending >> lane) & 1u) && digit == d;
    const unsigned group = __ballot_sync(0xffffffffu, mine);
    const uint32_t s0 = __reduce_add_sync(0xffffffffu, mine ? m0 : 0u);
    const uint32_t s1 = __reduce_add_sync(0xffffffffu, mine ? m1 : 0u);
    const uint32_t s2 = __reduce_add_sync(0xffffffffu, mine ? m2 : 0u);
    if (lane == leader) {
      atomicAdd(&h.p[0][d], s0);
      atomicAdd(&h.p[1][d], s1);
      atomicAdd(&h.p[2][d], s2);
      atomicAdd(&h.c[d], uint32_t(__popc(group)));
    }
    pending &= ~group;
  }
  if ((pending >> lane) & 1u) {
    atomicAdd(&h.p[0][digit], m0);
    atomicAdd(&h.p[1][digit], m1);
    atomicAdd(&h.p[2][digit], m2);
    atomicAdd(&h.c[digit], 1u);
  }
}

// Ranks candidate blocks by counting: candidate t (block cand[t], or block t
// without a list) is kept when the mass ranked before it (score desc, index
// asc) is below the target: `above` (every block ranked before all the
// candidates) plus the candidates ranked before it.  Thread t handles
// candidate t (nc <= kCountSel <= the CTA's threads).
template <bool kList>
__device__ __forceinline__ void rank_candidates(const SelectScratch& sc, const int* cand, int nc,
                                                unsigned long long above, unsigned long long target) {
  const int t = threadIdx.x;
  if (t >= nc) return;
  const int i = kList ? cand[t] : t;
  const unsigned long long ki = ((unsigned long long)sc.bits[i] << 32) | (0xFFFFFFFFu - uint32_t(i));
  unsigned long long before = above;
  for (int c = 0; c < nc; ++c) {
    const int j = kList ? cand[c] : c;
    const unsigned long long kj = ((unsigned long long)sc.bits[j] << 32) | (0xFFFFFFFFu - uint32_t(j));
    if (kj > ki) before += sc.m[j];
  }
  if (before < target) sc.keep[i] = 1;
}

// Selects the blocks of one request, called by every thread of a CTA of
// exactly kSelThreads threads: block scores bs[0..nb) (global, any state
// space the CTA can read), L tokens.  On return (after a barrier)
// sc.keep[i] says whether block i is kept (top-p set or exempt) and the
// kept-token count is returned to every thread.  A NaN, infinite or negative
// score keeps the whole request and records UPF_ERR_NONFINITE.
static __device__ int select_request(const float* bs, int nb, int L, int G, float top_p, int sink_keep, int tail_keep,
                              const SelectScratch& sc, int32_t* status) {
  __shared__ MassHist h_mass[2];   // this round's histogram and the next one's, cleared meanwhile
  __shared__ unsigned long long s_u64[kSelWarps];
  __shared__ float s_f[kSelWarps];
  __shared__ int s_i[kSelWarps];
  __shared__ int s_digit, s_count, s_ncand;
  __shared__ int s_cand[kCountSel];
  __shared__ unsigned long long s_above, s_wtot[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Load, validate (finite and >= 0) and find the largest score.
  float vmax = 0.f;
  int bad = 0;
  for (int i = tid; i < nb; i += blockDim.x) {
    const float v = __ldcg(bs + i);
    bad |= !(isfinite(v) && v >= 0.f);
    sc.bits[i] = __float_as_uint(v);
    vmax = fmaxf(vmax, v);
    sc.keep[i] = 0;
  }
  for (int d = tid; d < kHistWords; d += blockDim.x) (&h_mass[0].p[0][0])[d] = 0;   // the first round's histogram
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    s_f[warp] = vmax;
    s_i[warp] = bad;
  }
  __syncthreads();
  // Every per-warp maximum is a finite non-negative float unless `bad` is
  // set (then vmax is not used), so its bit pattern orders like its value.
  {
    const uint32_t fb = __float_as_uint(s_f[lane]);
    vmax = __uint_as_float(__reduce_max_sync(0xffffffffu, (fb & 0x80000000u) ? 0u : fb));
    bad = int(__reduce_or_sync(0xffffffffu, uint32_t(s_i[lane])));
  }
  if (bad) {
    if (tid == 0) set_status(status, UPF_ERR_NONFINITE);
    for (int i = tid; i < nb; i += blockDim.x) sc.keep[i] = 1;
  } else {
    int ex = 0;
    if (vmax > 0.f) frexpf(vmax, &ex);
    const int sh = 48 - ex;
    unsigned long long part = 0;
    for (int i = tid; i < nb; i += blockDim.x) {
      const unsigned long long m = vmax > 0.f ? fixed_mass(__uint_as_float(sc.bits[i]), sh) : 0ull;
      sc.m[i] = m;
      part += m;
    }
    // Mass the selected prefix must reach: the smallest integer >= top_p *
    // total (zero: no block by top-p).
    unsigned long long target = 0;
    if (nb <= kCountSel) {
      // Small request: every block is a candidate, ranked by counting (the
      // radix select's set, without its rounds and barriers).
      target = mass_target(top_p, sel_block_sum(part, s_u64));
      if (target > 0) rank_candidates<false>(sc, nullptr, nb, 0ull, target);
    } else {
      // The total comes out of the first round's bucket scan (every block is
      // in that round's histogram).
      uint32_t prefix = 0, pmask = 0;
      unsigned long long above = 0;   // mass of blocks ranked strictly before the candidates
      const int nb_pad = (nb + 31) & ~31;   // whole warps take part in the aggregation
      int cur = 0;
      bool few = false;   // the boundary bucket holds at most kCountSel blocks
      for (int shift = 24; shift >= 0; shift -= 8, cur ^= 1) {
        MassHist& hist = h_mass[cur];
        for (int i = tid; i < nb_pad; i += blockDim.x) {
          uint32_t digit = 256u + lane;        // nothing to add
          unsigned long long m = 0;
          if (i < nb) {
            const uint32_t b = sc.bits[i];
            if ((b & pmask) == prefix) {
              digit = (b >> shift) & 255u;
              m = sc.m[i];
            }
          }
          hist_add_aggregated(hist, digit, m);
        }
        __syncthreads();
        // Warps 0-7 scan the buckets from the highest digit down, 32 each
        // (lane l of warp w holds digit 255 - 32 w - l); the others clear the
        // next round's histogram.
        const int dg = 255 - 32 * warp - lane;
        unsigned long long mass = 0, incl = 0;
        if (warp < 8) {
          mass = hist_mass(hist, dg);
          incl = mass;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          if (lane == 31) s_wtot[warp] = incl;
        } else {
          for (int d = tid - 256; d < kHistWords; d += blockDim.x - 256)
            (&h_mass[cur ^ 1].p[0][0])[d] = 0;
          if (tid == 256) s_ncand = 0;
        }
        __syncthreads();
        if (shift == 24) {
          target = mass_target(top_p, warp_sum_u64(lane < 8 ? s_wtot[lane] : 0ull));
          if (target == 0) break;   // the same in every thread
        }
        if (warp < 8) {
          // Mass before this digit; exactly one digit starts below the target
          // and reaches it (the prefix bucket reaches it).
          const unsigned long long base = above + warp_sum_u64(lane < warp ? s_wtot[lane] : 0ull) + incl - mass;
          if (base < target && base + mass >= target) {
            s_digit = dg;
            s_above = base;
            s_count = int(hist.c[dg]);
          }
        }
        __syncthreads();
        prefix |= uint32_t(s_digit) << shift;
        pmask |= 255u << shift;
        above = s_above;
        // s_wtot, s_digit, s_above and s_count are rewritten only after the
        // next round's first barrier, which every thread reaches after
        // reading them here.
        if (s_count <= kCountSel) {
          few = true;
          break;
        }
      }
      if (few) {
        // Blocks above the boundary bucket are in; the bucket's blocks are
        // listed (in any order) and ranked by counting.  The same set as
        // finishing the rounds and taking ties in index order.
        for (int i = tid; i < nb_pad; i += blockDim.x) {
          bool cand = false;
          if (i < nb) {
            const uint32_t bm = sc.bits[i] & pmask;
            if (bm > prefix) sc.keep[i] = 1;
            cand = bm == prefix;
          }
          const unsigned bal = __ballot_sync(0xffffffffu, cand);
          if (bal) {
            int pos = 0;
            if (lane == 0) pos = atomicAdd(&s_ncand, __popc(bal));
            pos = __shfl_sync(0xffffffffu, pos, 0) + __popc(bal & ((1u << lane) - 1u));
            if (cand && pos < kCountSel) s_cand[pos] = i;
          }
        }
        __syncthreads();
        rank_candidates<true>(sc, s_cand, min(s_ncand, kCountSel), above, target);
      } else if (target > 0) {
        // prefix = bits of the boundary score v*.  Blocks above it are in; the
        // tied ones (equal scores) enter in index order until the mass suffices.
        // Thread t owns the contiguous index range [t*per, (t+1)*per).
        const int per = (nb + blockDim.x - 1) / blockDim.x;
        const int i0 = min(nb, tid * per), i1 = min(nb, i0 + per);
        int ties = 0;
        unsigned long long w = 0;
        for (int i = i0; i < i1; ++i) {
          const uint32_t b = sc.bits[i];
          if (b > prefix) sc.keep[i] = 1;
          else if (b == prefix) {
            ++ties;
            w = sc.m[i];
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
        const int before = incl - ties + warps_before_sum(s_i);
        if (ties > 0) {
          // every tied block carries the same mass w > 0 (the boundary bucket reached the target)
          const unsigned long long need = target - above;   // > 0: the boundary bucket is needed
          // Usually one tied block suffices (need <= w); the division is for the rest.
          const unsigned long long take = need <= w ? 1ull : (w > 0 ? (need + w - 1) / w : 0ull);
          int rank = before;
          for (int i = i0; i < i1; ++i)
            if (sc.bits[i] == prefix) {
              if ((unsigned long long)rank < take) sc.keep[i] = 1;
              ++rank;
            }
        }
      }
    }
  }
  __syncthreads();
  // Exempt blocks (overlap with [0, sink) or [L - tail, L)) and the kept
  // tokens, each block by the thread that owns it in this loop.
  const int sink_hi = min(sink_keep, L);
  const int tail_lo = max(0, L - tail_keep);
  __shared__ int s_cw[kSelWarps];
  int cnt = 0;
  for (int i = tid; i < nb; i += blockDim.x) {
    const int lo = i * G, hi = min(L, lo + G);
    bool kept = sc.keep[i] != 0;
    if (lo < sink_hi || hi > tail_lo) {
      sc.keep[i] = 1;
      kept = true;
    }
    if (kept) cnt += hi - lo;
  }
  cnt = int(__reduce_add_sync(0xffffffffu, uint32_t(cnt)));
  if (lane == 0) s_cw[warp] = cnt;
  __syncthreads();
  return int(__reduce_add_sync(0xffffffffu, uint32_t(s_cw[lane])));
}

// Keep-bit word w of the packed tokens [tok0, tok0 + L) of a request whose
// block flags are keep[]: bit (t % 32) set for kept tokens t of the request
// in that word, 0 for tokens outside it.  gshift = log2(G) when G is a power
// of two (the block of a token is then a shift), else -1.
__device__ __forceinline__ uint32_t request_word_bits(const unsigned char* keep, int tok0, int L, int G, int gshift,
                                                      int w) {
  if (gshift >= 5 && (tok0 & 31) == 0) {
    // Blocks are whole words: the word's tokens share one block (the last
    // word of the request may hold fewer than 32 of its tokens).
    const int t = w * 32, n = min(32, tok0 + L - t);
    return keep[(t - tok0) >> gshift] ? (n >= 32 ? 0xffffffffu : ((1u << n) - 1u)) : 0u;
  }
  uint32_t bits = 0;
  const int t_lo = max(tok0, w * 32), t_hi = min(tok0 + L, w * 32 + 32);
  for (int t = t_lo; t < t_hi;) {   // walk the blocks that overlap this word's tokens
    const int blk = gshift >= 0 ? (t - tok0) >> gshift : (t - tok0) / G;
    const int t_end = min(t_hi, tok0 + (blk + 1) * G);
    if (keep[blk]) {
      const int len = t_end - t;
      bits |= (len >= 32 ? 0xffffffffu : ((1u << len) - 1u)) << (t & 31);
    }
    t = t_end;
  }
  return bits;
}

__host__ __device__ __forceinline__ int block_shift(int G) {
  if (G <= 0 || (G & (G - 1))) return -1;
  int k = 0;
  while ((1 << k) < G) ++k;
  return k;
}

}  // namespace upf
