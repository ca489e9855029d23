// pkv_plan.cuh -- the device-side plan of a decode step, shared by the SIMT
// and the tensor-core decode kernels.
//
// The step's decode work is the sequence of row-groups (query row, KV head)
// in request order, each a run of 16-token blocks: row i of request r (q_r
// query tokens, length L) sees positions < L - q_r + i + 1 (the chunk sits at
// the end of the sequence: The Serving Playbook, "Chunked prefill").  The
// grid cuts that block sequence into equal contiguous ranges, one per CTA,
// so every CTA streams the same number of tiles whatever the length mix; a
// row-group cut by a range boundary is computed in pieces that are merged by
// log-sum-exp (The Serving Playbook, "Kernel fusion, briefly": Flash-Decoding
// splits the KV axis).
//
// One warp of each CTA computes the plan from seq_lens / query_start_loc in
// device memory (a warp-wide scan over the requests), so the launch shape
// depends only on bounds and the call can be captured in a CUDA graph.
#pragma once

#include <climits>

#include "pkv_internal.h"

namespace pkv {
namespace plan {

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }
__device__ __forceinline__ long long cdiv_ll(long long a, long long b) { return (a + b - 1) / b; }

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

__device__ __forceinline__ ReqInfo load_request(const DecodeParams& p, int r) {
  ReqInfo ri;
  ri.q0 = __ldg(p.qsl + r);
  const int q1 = __ldg(p.qsl + r + 1);
  ri.L = __ldg(p.seq_lens + r);
  ri.qr = q1 - ri.q0;
  const bool ok = ri.q0 >= 0 && ri.qr >= 0 && q1 <= p.num_q_tokens && ri.qr <= ri.L &&
                  ri.L <= p.max_blocks * kBlockSize;
  ri.decode = ok && ri.qr > 0 && ri.qr < p.prefill_min_q;
  // A shared prefix (cascade) must end before the request's first query.
  ri.fb = p.first_block ? __ldg(p.first_block + r) : 0;
  if (ri.fb < 0 || (long long)ri.fb * kBlockSize > (long long)ri.L - ri.qr) ri.fb = 0;
  return ri;
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

// This CTA's share [lo, hi) of the step's block sequence, and the range
// length (chunk) every CTA uses.  Warp-collective.
struct Range {
  long long lo, hi, chunk;
};

__device__ __forceinline__ Range cta_range(const DecodeParams& p, int lane) {
  const int R = p.num_reqs, Hkv = p.num_kv_heads;
  long long mine = 0;
  int nb_min = INT_MAX, nb_max = 0;
  for (int r = lane; r < R; r += 32) {
    const ReqInfo ri = load_request(p, r);
    if (ri.decode) {
      mine += rows_blocks(ri, ri.qr) * Hkv;
      nb_min = min(nb_min, row_blocks(ri, 0));
      nb_max = max(nb_max, row_blocks(ri, ri.qr - 1));
    } else if (blockIdx.x == 0 && ri.qr != 0 && ri.qr < p.prefill_min_q) {
      record_error(p.err, kErrBounds);  // inconsistent lengths: request skipped
    }
  }
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
    nb_min = min(nb_min, __shfl_xor_sync(0xffffffffu, nb_min, o));
    nb_max = max(nb_max, __shfl_xor_sync(0xffffffffu, nb_max, o));
  }
  const long long W = mine;
  long long chunk = max((long long)p.min_chunk, cdiv_ll(W, gridDim.x));
  if (p.align && nb_min == nb_max && W > 0) {
    // Uniform row-groups: cut each into equal pieces, or keep whole groups
    // together, so that piece boundaries coincide with CTA boundaries --
    // unless that lengthens every CTA's range by more than align_slack
    // blocks (then idle CTAs cost more than the extra pieces save).
    const long long nb = nb_max;
    const long long snapped = chunk < nb ? cdiv_ll(nb, nb / chunk) : cdiv_ll(chunk, nb) * nb;
    if (snapped - chunk <= p.align_slack) chunk = snapped;
  }
  Range rg;
  rg.chunk = chunk;
  rg.lo = (long long)blockIdx.x * chunk;
  rg.hi = min(W, rg.lo + chunk);
  return rg;
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
        if (q.decode) w = rows_blocks(q, q.qr) * Hkv;
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
    ri = load_request(p, r);
    {  // first row of request r whose groups reach lo (binary search)
      int a = 0, b = ri.qr - 1;
      while (a < b) {
        const int mid = (a + b + 1) / 2;
        if (pos + rows_blocks(ri, mid) * Hkv <= rg.lo) a = mid; else b = mid - 1;
      }
      i = a;
    }
    g = pos + rows_blocks(ri, i) * Hkv;  // start of row i, head 0
    nb = row_blocks(ri, i);
    k = (int)((rg.lo - g) / nb);
    g += (long long)k * nb;
    done = g >= rg.hi;
  }

  // The current piece, then advance.  False when the range is exhausted.
  __device__ __forceinline__ bool next(const DecodeParams& p, Piece& pc) {
    if (done) return false;
    const long long s0 = max(g, rg.lo), s1 = min(g + nb, rg.hi);
    const long long c0 = g / rg.chunk, c1 = (g + nb - 1) / rg.chunk;
    pc.row = ri.q0 + i;
    pc.r = r;
    pc.k = k;
    pc.b0 = ri.fb + (int)(s0 - g);
    pc.pre = ri.fb > 0;
    pc.fb = ri.fb;
    pc.nblk = (int)(s1 - s0);
    pc.limit = ri.L - ri.qr + i + 1;
    pc.L = ri.L;
    pc.S = (int)(c1 - c0 + 1);
    pc.c0 = (int)c0;
    pc.odd0 = g != c0 * rg.chunk;
    pc.slot = 2 * (int)blockIdx.x + (s0 == rg.lo ? 0 : 1);
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
      if (!done) nb = row_blocks(ri, i);
    }
    if (g >= rg.hi) done = true;
    return true;
  }
};

// Warms L2 with the part of the block table this CTA will probably read (its
// share of the step if every row were full).
__device__ __forceinline__ void prefetch_block_table(const DecodeParams& p, int lane) {
  const long long entries = (long long)p.num_reqs * p.max_blocks;
  const long long est = entries * blockIdx.x / gridDim.x;
  const long long line0 = (est * 4) / 128 - 2;
  const long long lines = (entries * 4 + 127) / 128;
  const long long line = line0 + lane;
  if (line >= 0 && line < lines)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.block_tables) +
                                                 line * 128));
}

}  // namespace plan
}  // namespace pkv
