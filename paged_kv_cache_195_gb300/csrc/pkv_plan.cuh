// pkv_plan.cuh -- the device-side plan of a decode step, shared by the SIMT
// and the tensor-core decode kernels.
//
// The step's decode work is the sequence of row-groups (query row, KV head)
// in request order, each a run of 16-token blocks: row i of request r (q_r
// query tokens, length L) sees positions < L - q_r + i + 1 (the chunk sits at
// the end of the sequence: The Serving Playbook, "Chunked prefill").  The
// grid cuts that block sequence into equal contiguous ranges, one per CTA --
// over weighted lengths, each row-group counting a few blocks more for the
// fixed cost of a piece -- so every CTA has about the same work whatever the
// length mix; a row-group cut by a range boundary is computed in pieces that
// are merged by log-sum-exp (The Serving Playbook, "Kernel fusion, briefly":
// Flash-Decoding splits the KV axis).
//
// One warp of each CTA computes the plan from seq_lens / query_start_loc in
// device memory (a warp-wide scan over the requests), so the launch shape
// depends only on bounds and the call can be captured in a CUDA graph.  For
// steps of up to 256 requests each CTA also keeps its plan in the workspace,
// with the exact inputs it came from, and reuses it while they are unchanged
// (every layer of an engine step has the same lengths).
#pragma once

#include <climits>

#include "pkv_internal.h"

namespace pkv {
namespace plan {

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }
// a / b for a >= 0, b > 0: a 32-bit division whenever both fit (the usual
// case; a 64-bit division is several times longer).
__device__ __forceinline__ long long div_ll(long long a, long long b) {
  if ((unsigned long long)(a | b) <= 0xffffffffull) return (unsigned)a / (unsigned)b;
  return a / b;
}
__device__ __forceinline__ long long cdiv_ll(long long a, long long b) { return div_ll(a + b - 1, b); }

// Sum over x = 1..n of ceil(x / 16): with n = 16m + t, 8m(m+1) + t(m+1).
__device__ __forceinline__ long long ceil16_prefix(long long n) {
  if (n <= 0) return 0;
  const long long m = n / kBlockSize, t = n % kBlockSize;
  return 8 * m * (m + 1) + t * (m + 1);
}

struct ReqInfo {
  int q0, qr, L;
  int fb;       // first block this call reads (a shared prefix before it is computed elsewhere)
  bool decode;  // has rows the decode kernels serve
};

// A request's record from its raw fields (query_start_loc[r], [r + 1],
// seq_lens[r], first_block[r]).
__device__ __forceinline__ ReqInfo make_request(const DecodeParams& p, int q0, int q1, int L,
                                                int fb) {
  ReqInfo ri;
  ri.q0 = q0;
  ri.L = L;
  ri.qr = q1 - q0;
  const bool ok = ri.q0 >= 0 && ri.qr >= 0 && q1 <= p.num_q_tokens && ri.qr <= ri.L &&
                  ri.L <= p.max_blocks * kBlockSize;
  ri.decode = ok && ri.qr > 0 && ri.qr < p.prefill_min_q;
  // A shared prefix (cascade) must end before the request's first query.
  ri.fb = fb;
  if (ri.fb < 0 || (long long)ri.fb * kBlockSize > (long long)ri.L - ri.qr) ri.fb = 0;
  return ri;
}

__device__ __forceinline__ ReqInfo load_request(const DecodeParams& p, int r) {
  return make_request(p, __ldg(p.qsl + r), __ldg(p.qsl + r + 1), __ldg(p.seq_lens + r),
                      p.first_block ? __ldg(p.first_block + r) : 0);
}

// Blocks row i reads: positions fb*16 .. L - qr + i (row i sees L - qr + i + 1 keys).
__device__ __forceinline__ int row_blocks(const ReqInfo& ri, int i) {
  return cdiv(ri.L - ri.qr + i + 1, kBlockSize) - ri.fb;
}

// Blocks of rows 0..i-1 of a request (one KV head).
__device__ __forceinline__ long long rows_blocks(const ReqInfo& ri, int i) {
  const long long a = (long long)ri.L - ri.qr + 1;
  return ceil16_prefix(a + i - 1) - ceil16_prefix(a - 1) - (long long)i * ri.fb;
}

// The ranges are cut over weighted lengths: each row-group counts as its
// blocks plus p.rowgroup_cost, the fixed cost of a piece (its epilogue, its
// last partial tile) in blocks' worth of streaming, so that a CTA whose range
// holds many short row-groups gets fewer blocks.  The weight's extra units
// sit after the row-group's real blocks and hold no work.
__device__ __forceinline__ int row_weight(const DecodeParams& p, const ReqInfo& ri, int i) {
  return row_blocks(ri, i) + p.rowgroup_cost;
}

// Weighted length of rows 0..i-1 of a request (one KV head).
__device__ __forceinline__ long long rows_weight(const DecodeParams& p, const ReqInfo& ri, int i) {
  return rows_blocks(ri, i) + (long long)i * p.rowgroup_cost;
}

// This CTA's share [lo, hi) of the step's weighted block sequence, and the
// range length (chunk) every CTA uses.  Warp-collective.
struct Range {
  long long lo, hi, chunk;
};

// Adds request r's row-groups to this lane's running totals (its blocks over
// all rows and KV heads, the extreme row-group lengths); returns its blocks.
__device__ __forceinline__ long long tally_request(const DecodeParams& p, const ReqInfo& ri, int r,
                                                   long long& mine, int& nb_min, int& nb_max) {
  long long w = 0;
  if (ri.decode) {
    w = rows_weight(p, ri, ri.qr) * p.num_kv_heads;
    nb_min = min(nb_min, row_weight(p, ri, 0));
    nb_max = max(nb_max, row_weight(p, ri, ri.qr - 1));
  } else if (blockIdx.x == 0 && r < p.num_reqs && ri.qr != 0 && ri.qr < p.prefill_min_q) {
    record_error(p.err, kErrBounds);  // inconsistent lengths: request skipped
  }
  mine += w;
  return w;
}

// The range from the lanes' totals.  Warp-collective.
__device__ __forceinline__ Range finish_range(const DecodeParams& p, long long mine, int nb_min,
                                              int nb_max) {
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
    nb_min = min(nb_min, __shfl_xor_sync(0xffffffffu, nb_min, o));
    nb_max = max(nb_max, __shfl_xor_sync(0xffffffffu, nb_max, o));
  }
  const long long W = mine;
  // Steps with little work run on the first half of the grid (one CTA per
  // SM when the grid is two per SM), leaving each SM's second slot to the
  // next launch, which can then prepare while this one streams.
  const int ctas = p.half_grid_blocks > 0 && W <= (long long)p.half_grid_blocks * (gridDim.x / 2)
                       ? (int)(gridDim.x / 2) : (int)gridDim.x;
  long long chunk = max((long long)p.min_chunk, cdiv_ll(W, ctas));
  if (p.align && nb_min == nb_max && W > 0) {
    // Uniform row-groups: cut each into equal pieces, or keep whole groups
    // together, so that piece boundaries coincide with CTA boundaries --
    // unless that lengthens every CTA's range by more than align_slack
    // blocks (then idle CTAs cost more than the extra pieces save).
    const long long nb = nb_max;
    const long long snapped = chunk < nb ? cdiv_ll(nb, div_ll(nb, chunk)) : cdiv_ll(chunk, nb) * nb;
    if (snapped - chunk <= p.align_slack) chunk = snapped;
  }
  Range rg;
  rg.chunk = chunk;
  rg.lo = (long long)blockIdx.x * chunk;
  rg.hi = min(W, rg.lo + chunk);
  return rg;
}

__device__ __forceinline__ Range cta_range(const DecodeParams& p, int lane) {
  long long mine = 0;
  int nb_min = INT_MAX, nb_max = 0;
  for (int r = lane; r < p.num_reqs; r += 32)
    tally_request(p, load_request(p, r), r, mine, nb_min, nb_max);
  return finish_range(p, mine, nb_min, nb_max);
}

// One piece of a row-group: the blocks [b0, b0 + nblk) of row `row`, KV head k.
struct Piece {
  int row;     // global query row, or kEndRow
  int r;       // request
  int k;       // KV head
  int b0;      // first logical block of the piece (a table column)
  int pre;     // the row's shared prefix was computed by the prefix pass (merge it)
  int fb;      // shared blocks before the row's own (the prefix pass covered them)
  int nblk;    // blocks in the piece (>= 1)
  int limit;   // keys visible to this row: positions < limit
  int L;       // request length (positions >= L hold no key)
  int fresh;   // first table column holding one of this step's new tokens
  int slot;    // workspace slot of this piece's partial state (partial pieces)
  int c0;      // first CTA whose range touches the row-group
  int S;       // pieces of the row-group (1: complete in this CTA)
  int odd0;    // piece 0 of the row-group uses slot 2*c0+1 (else 2*c0)
};
constexpr int kEndRow = -2;  // piece marker: the CTA's range is done

// Walks the pieces of the row-groups that intersect [lo, hi), in order.
// Warp-collective; every lane holds the same state.
struct Walker {
  Range rg;
  long long g;  // first global block of the current row-group
  int r, i, k, nb;
  ReqInfo ri;
  bool done;

  // Finds the request and row that hold block lo (a warp-wide scan).
  __device__ __forceinline__ void start(const DecodeParams& p, const Range& range, int lane) {
    rg = range;
    done = rg.lo >= rg.hi;
    if (done) return;
    const int R = p.num_reqs, Hkv = p.num_kv_heads;
    r = -1;
    long long pos = 0, base = 0;
    for (int b = 0; b < R; b += 32) {
      const int rr = b + lane;
      long long w = 0;
      if (rr < R) {
        const ReqInfo q = load_request(p, rr);
        if (q.decode) w = rows_weight(p, q, q.qr) * Hkv;
      }
      long long incl = w;
      #pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const long long excl = incl - w;
      const unsigned own =
          __ballot_sync(0xffffffffu, w > 0 && base + excl <= rg.lo && rg.lo < base + incl);
      if (own) {
        const int src = __ffs(own) - 1;
        r = b + src;
        pos = base + __shfl_sync(0xffffffffu, excl, src);
        break;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (r < 0) {
      record_error(p.err, kErrBounds);  // unreachable when the lengths are stable
      done = true;
      return;
    }
    finish_start(p, load_request(p, r), pos);
  }

  // Request r (record q, first global block pos) holds block lo: the row,
  // KV head and row-group the range starts in.
  __device__ __forceinline__ void finish_start(const DecodeParams& p, const ReqInfo& q,
                                               long long pos) {
    const int Hkv = p.num_kv_heads;
    ri = q;
    {  // first row of request r whose groups reach lo (binary search)
      int a = 0, b = ri.qr - 1;
      while (a < b) {
        const int mid = (a + b + 1) / 2;
        if (pos + rows_weight(p, ri, mid) * Hkv <= rg.lo) a = mid; else b = mid - 1;
      }
      i = a;
    }
    g = pos + rows_weight(p, ri, i) * Hkv;  // start of row i, head 0
    nb = row_weight(p, ri, i);
    k = (int)div_ll(rg.lo - g, nb);
    g += (long long)k * nb;
    done = g >= rg.hi;
  }

  // The next piece of the range, then advance.  False when the range is
  // exhausted.  A row-group's real blocks are [g, g + nb - rowgroup_cost) of
  // its weighted extent [g, g + nb); a range that meets only the rest of it
  // has no piece of that row-group.
  __device__ __forceinline__ bool next(const DecodeParams& p, Piece& pc) {
    while (!done) {
      const long long nbr = nb - p.rowgroup_cost;  // real blocks
      const long long s0 = max(g, rg.lo), s1 = min(g + nbr, rg.hi);
      const bool emit = s0 < s1;
      if (emit) {
        const long long c0 = div_ll(g, rg.chunk), c1 = div_ll(g + nbr - 1, rg.chunk);
        pc.row = ri.q0 + i;
        pc.r = r;
        pc.k = k;
        pc.b0 = ri.fb + (int)(s0 - g);
        pc.pre = ri.fb > 0;
        pc.fb = ri.fb;
        pc.nblk = (int)(s1 - s0);
        pc.limit = ri.L - ri.qr + i + 1;
        pc.L = ri.L;
        pc.fresh = (ri.L - ri.qr) / kBlockSize;
        pc.S = (int)(c1 - c0 + 1);
        pc.c0 = (int)c0;
        pc.odd0 = g != c0 * rg.chunk;
        pc.slot = 2 * (int)blockIdx.x + (s0 == rg.lo ? 0 : 1);
      }
      // advance to the next row-group
      g += nb;
      if (++k == p.num_kv_heads) {
        k = 0;
        if (++i == ri.qr) {
          i = 0;
          do {
            ++r;
            if (r >= p.num_reqs) break;
            ri = load_request(p, r);
          } while (!ri.decode);
          if (r >= p.num_reqs) done = true;
        }
        if (!done) nb = row_weight(p, ri, i);
      }
      if (g >= rg.hi) done = true;
      if (emit) return true;
    }
    return false;
  }
};

// Requests per lane whose records plan_cta keeps in registers: steps of up to
// 32 * kPlanRegReqs requests are planned from one batch of loads.
constexpr int kPlanRegReqs = 8;
static_assert(32 * kPlanRegReqs <= kPlanCacheReqs, "plan cache too small");

// Plan cache entry (one per CTA index, int32 words): the inputs the plan was
// computed from -- a header of sizes and tuning values, query_start_loc and
// seq_lens -- and the resulting range and walker state.  Every layer of an
// engine step has the same lengths, so a CTA computes its plan once per step
// and later calls compare and reuse it; the comparison is exact, so a reused
// plan is always the plan of the current lengths.
constexpr int kPcHeader = 11, kPcQsl = 16, kPcLens = kPcQsl + kPlanCacheReqs + 4,
              kPcState = kPcLens + kPlanCacheReqs, kPcStateWords = 18;
static_assert(kPcState + kPcStateWords <= kPlanEntryWords, "plan cache entry layout");
constexpr int kPcMagic = 0x504c414e;

__device__ __forceinline__ int plan_header_word(const DecodeParams& p, int j) {
  switch (j) {
    case 0: return p.num_reqs;
    case 1: return p.num_q_tokens;
    case 2: return p.num_kv_heads;
    case 3: return p.prefill_min_q;
    case 4: return p.min_chunk;
    case 5: return p.align;
    case 6: return p.align_slack;
    case 7: return (int)gridDim.x;
    case 8: return p.max_blocks;
    case 9: return p.rowgroup_cost;
    default: return kPcMagic ^ p.half_grid_blocks;
  }
}

// The CTA's range and a walker at its first row-group: the same result as
// cta_range followed by Walker::start, but for steps of up to 32 *
// kPlanRegReqs requests every record is loaded once, all loads are in flight
// together, and each lane takes a contiguous run of requests so that one
// warp-wide scan finds the request holding the range's first block.
// Warp-collective.
__device__ __forceinline__ void plan_cta(const DecodeParams& p, int lane, Range& rg,
                                         Walker& wk) {
  const int R = p.num_reqs;
  if (R > 32 * kPlanRegReqs) {
    rg = cta_range(p, lane);
    wk.start(p, rg, lane);
    return;
  }
  const int per = (R + 31) / 32;  // requests per lane: r0 .. r0 + per - 1
  const int r0 = lane * per;
  // The cached plan of this CTA index, if any (not for shared-prefix calls,
  // whose first blocks change with every call).
  int* const ce = p.plan_cache != nullptr && p.first_block == nullptr &&
                          (int)blockIdx.x < p.plan_entries
                      ? p.plan_cache + (long long)blockIdx.x * kPlanEntryWords
                      : nullptr;
  int a0[kPlanRegReqs], a1[kPlanRegReqs], aL[kPlanRegReqs], aF[kPlanRegReqs];
  int c0[kPlanRegReqs], c1[kPlanRegReqs], cL[kPlanRegReqs];
  int ch = 0, cs = 0;
  if (ce != nullptr) {  // issued together with the request loads below
    if (lane < kPcHeader) ch = __ldcg(ce + lane);
    if (lane < kPcStateWords) cs = __ldcg(ce + kPcState + lane);
  }
  #pragma unroll
  for (int i = 0; i < kPlanRegReqs; ++i) {
    const int r = r0 + i;
    const bool in = i < per && r < R;
    a0[i] = in ? __ldg(p.qsl + r) : 0;
    a1[i] = in ? __ldg(p.qsl + r + 1) : 0;
    aL[i] = in ? __ldg(p.seq_lens + r) : 0;
    aF[i] = in && p.first_block ? __ldg(p.first_block + r) : 0;
    const bool cin = in && ce != nullptr;
    c0[i] = cin ? __ldcg(ce + kPcQsl + r) : 0;
    c1[i] = cin ? __ldcg(ce + kPcQsl + r + 1) : 0;
    cL[i] = cin ? __ldcg(ce + kPcLens + r) : 0;
  }
  if (ce != nullptr) {
    bool same = lane >= kPcHeader || ch == plan_header_word(p, lane);
    #pragma unroll
    for (int i = 0; i < kPlanRegReqs; ++i)
      same = same && (i >= per || (a0[i] == c0[i] && a1[i] == c1[i] && aL[i] == cL[i]));
    if (__all_sync(0xffffffffu, same)) {
      auto word = [&](int j) { return __shfl_sync(0xffffffffu, cs, j); };
      auto dword = [&](int j) {
        return (long long)(((unsigned long long)(unsigned)word(j + 1) << 32) | (unsigned)word(j));
      };
      rg.lo = dword(0);
      rg.hi = dword(2);
      rg.chunk = dword(4);
      wk.rg = rg;
      wk.g = dword(6);
      wk.r = word(8);
      wk.i = word(9);
      wk.k = word(10);
      wk.nb = word(11);
      wk.done = word(12) != 0;
      wk.ri.q0 = word(13);
      wk.ri.qr = word(14);
      wk.ri.L = word(15);
      wk.ri.fb = word(16);
      wk.ri.decode = word(17) != 0;
      return;
    }
  }
  // After computing: record the plan in the cache (the next calls with these
  // lengths reuse it).  Lanes that share a query_start_loc entry write the
  // same value.
  auto record = [&]() {
    if (ce == nullptr) return;
    #pragma unroll
    for (int i = 0; i < kPlanRegReqs; ++i) {
      const int r = r0 + i;
      if (i < per && r < R) {
        __stcg(ce + kPcQsl + r, a0[i]);
        __stcg(ce + kPcQsl + r + 1, a1[i]);
        __stcg(ce + kPcLens + r, aL[i]);
      }
    }
    int sv = 0;
    auto put = [&](int j, int v) { if (lane == j) sv = v; };
    auto put2 = [&](int j, long long v) {
      put(j, (int)(unsigned)(unsigned long long)v);
      put(j + 1, (int)(unsigned)((unsigned long long)v >> 32));
    };
    put2(0, wk.rg.lo);
    put2(2, wk.rg.hi);
    put2(4, wk.rg.chunk);
    put2(6, wk.g);
    put(8, wk.r);
    put(9, wk.i);
    put(10, wk.k);
    put(11, wk.nb);
    put(12, wk.done ? 1 : 0);
    put(13, wk.ri.q0);
    put(14, wk.ri.qr);
    put(15, wk.ri.L);
    put(16, wk.ri.fb);
    put(17, wk.ri.decode ? 1 : 0);
    if (lane < kPcStateWords) __stcg(ce + kPcState + lane, sv);
    if (lane < kPcHeader) __stcg(ce + lane, plan_header_word(p, lane));
    __threadfence();
  };
  long long w[kPlanRegReqs];
  long long mine = 0;
  int nb_min = INT_MAX, nb_max = 0;
  #pragma unroll
  for (int i = 0; i < kPlanRegReqs; ++i) {
    w[i] = 0;
    if (i < per) {  // warp-uniform: the iterations past the runs are skipped
      const int r = r0 + i;
      ReqInfo q = make_request(p, a0[i], a1[i], aL[i], aF[i]);
      q.decode = q.decode && r < R;
      w[i] = tally_request(p, q, r, mine, nb_min, nb_max);
    }
  }
  const long long own_total = mine;
  rg = finish_range(p, mine, nb_min, nb_max);
  wk.rg = rg;
  wk.done = rg.lo >= rg.hi;
  if (wk.done) {
    wk.g = 0;
    wk.r = wk.i = wk.k = wk.nb = 0;
    wk.ri = ReqInfo{0, 0, 0, 0, false};
    record();
    return;
  }
  // Blocks of the requests before this lane's run (exclusive scan).
  long long incl = own_total;
  #pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const long long base = incl - own_total;
  const unsigned own = __ballot_sync(0xffffffffu, own_total > 0 && base <= rg.lo && rg.lo < incl);
  if (own == 0) {
    record_error(p.err, kErrBounds);  // unreachable when the lengths are stable
    wk.done = true;
    return;
  }
  const int owner = __ffs(own) - 1;
  // The owner lane walks its run to the request that holds block lo.
  int fr = 0, f0 = 0, f1 = 0, fL = 0, fF = 0;
  long long pos = 0;
  if (lane == owner) {
    long long acc = base;
    bool found = false;
    #pragma unroll
    for (int i = 0; i < kPlanRegReqs; ++i) {
      if (i < per && !found && w[i] > 0 && rg.lo < acc + w[i]) {
        found = true;
        fr = r0 + i;
        f0 = a0[i];
        f1 = a1[i];
        fL = aL[i];
        fF = aF[i];
        pos = acc;
      }
      acc += w[i];
    }
  }
  fr = __shfl_sync(0xffffffffu, fr, owner);
  f0 = __shfl_sync(0xffffffffu, f0, owner);
  f1 = __shfl_sync(0xffffffffu, f1, owner);
  fL = __shfl_sync(0xffffffffu, fL, owner);
  fF = __shfl_sync(0xffffffffu, fF, owner);
  pos = __shfl_sync(0xffffffffu, pos, owner);
  wk.r = fr;
  wk.finish_start(p, make_request(p, f0, f1, fL, fF), pos);
  record();
}

}  // namespace plan
}  // namespace pkv
