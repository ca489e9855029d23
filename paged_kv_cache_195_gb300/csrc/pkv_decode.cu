// pkv_decode.cu -- paged decode attention with split context and a fused
// log-sum-exp merge, for sm_103a.
//
// What it computes (per query row t of request r, KV head k, and the g query
// heads h = k*g .. k*g+g-1 that share KV head k): the softmax-weighted sum of
// V over the keys the row may see, gathered block by block through the
// request's block table (The Serving Playbook, "The block table lives in the
// hottest kernel in the system").
//
// How, on GB300:
//  * One CTA serves all g query heads of a KV head, so each (block, KV head)
//    tile -- 4 KiB of K and 4 KiB of V, contiguous in the pool -- leaves HBM
//    once per row.
//  * Parallelism comes from the KV axis (Flash-Decoding: The Serving
//    Playbook, "Kernel fusion, briefly").  The step's work is the sequence of
//    (row, KV head) row-groups, each a run of 16-token blocks; a persistent
//    grid cuts that sequence into equal contiguous ranges, one per CTA, so
//    every CTA streams the same number of tiles whatever the length mix.  A
//    row-group cut by a range boundary is computed in pieces; each piece
//    keeps an online-softmax state (running max, normaliser, rescaled output:
//    LLM 7 - Efficient LLM Serving, sec. 2 "Online Softmax Makes Tiling
//    Possible"), and the last CTA to finish a row-group merges its pieces by
//    log-sum-exp, found with one atomic counter per row-group: no extra
//    launch, merge in piece order (deterministic).
//  * The plan -- the block count of every request, their prefix sum and this
//    CTA's range -- is computed by the producer warp of every CTA from
//    seq_lens / query_start_loc in device memory, so the launch shape depends
//    only on bounds and the call is CUDA-graph capturable.
//  * The producer warp walks the CTA's range and issues cp.async.bulk copies of
//    whole tiles into an 8-stage shared-memory ring (mbarrier-tracked), running
//    ahead across piece boundaries; four consumer warps take stages
//    round-robin.  Two CTAs per SM keep ~128 KiB of loads in flight per SM.
//  * Consumers: lane = (token half, 16-byte chunk of d).  q for all g heads of
//    the lane's chunk stays in registers; QK partial sums over the lane's 8
//    dims are reduced across the 16 lanes of a half-warp by a reduce-scatter
//    whose register order is permuted per lane so that no selects are needed;
//    softmax in fp32 (exp2 with scale*log2(e) folded into q); PV accumulates
//    in packed fp32 (fma.rn.f32x2).
#include <climits>
#include <cstdio>
#include <cstdlib>

#include "pkv_internal.h"

namespace pkv {
namespace {

// Warp layout.  Blocks are consumed by four warp groups in turn; with an
// even group size g the g query heads are split across the two warps of a
// group (each warp owns g/2 heads: half the registers, twice the warps per
// SM to hide latency), otherwise one warp holds all g heads.
#ifndef PKV_HSPLIT
#define PKV_HSPLIT 0
#endif
#ifndef PKV_GROUPS_SPLIT
#define PKV_GROUPS_SPLIT 3
#endif
template <int G>
struct DecodeCfg {
  static constexpr int kHS = (PKV_HSPLIT && G % 2 == 0) ? 2 : 1;  // warps per group
  static constexpr int kGH = G / kHS;                             // heads per warp
  static constexpr int kGroups = kHS == 2 ? PKV_GROUPS_SPLIT : 4;  // blocks in flight per round
  static constexpr int kCW = kGroups * kHS;                       // consumer warps
  static constexpr int kThreads = (kCW + 1) * 32;                 // + producer warp
  static constexpr int kMinCtas = (kGH <= 6) ? 2 : 1;
  // Registers per thread that still let kMinCtas CTAs share an SM (the
  // register file is handed out as if a CTA's warp count were even).
  static constexpr int kWarpsAlloc = (kCW + 2) / 2 * 2;
  static constexpr int kMaxRegs =
      kMinCtas == 1 ? 255 : (65536 / (kMinCtas * kWarpsAlloc * 32)) / 8 * 8;
};

// Ring depth: 8 stages per CTA when two CTAs share an SM (shared memory),
// 20 when one CTA has the SM to itself.
#ifndef PKV_RING
#define PKV_RING 8
#endif
template <int G>
constexpr int stages_for() { return DecodeCfg<G>::kMinCtas == 2 ? PKV_RING : 20; }
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr float kNegBig = -1.0e30f;          // "no key seen yet" running max
constexpr int kEndRow = -2;                  // piece marker: the CTA's range is done

// One piece of a row-group: the blocks [b0, b0 + nblk) of row `row`, KV head k.
struct Piece {
  int row;     // global query row, or kEndRow
  int k;       // KV head
  int b0;      // first logical block of the piece
  int nblk;    // blocks in the piece (>= 1)
  int limit;   // keys visible to this row: positions < limit
  int slot;    // workspace slot of this piece's partial state (partial pieces)
  int c0;      // first CTA whose range touches the row-group
  int S;       // pieces of the row-group (1: complete in this CTA)
  int odd0;    // piece 0 of the row-group uses slot 2*c0+1 (else 2*c0)
};

#ifndef PKV_P_DUP
#define PKV_P_DUP 0
#endif

template <int G>
struct __align__(128) DecodeSmem {
  using Cfg = DecodeCfg<G>;
  static constexpr int kStages = stages_for<G>();
  // Probabilities of one block, stored twice ({p, p}) so that the PV loop
  // feeds packed fp32 FMAs straight from 16-byte loads.
#if PKV_P_DUP
  static constexpr int kPStride = (Cfg::kGH + 1) & ~1;  // float2 entries per token
#else
  static constexpr int kPStride = ((Cfg::kGH + 3) & ~3) / 2;  // float2 slots = 2 floats each
#endif
  uint8_t ring[kStages][kStageBytes];
  __nv_bfloat16 qbuf[2][G * kHeadDim];
  float2 pbuf[Cfg::kCW][kBlockSize][kPStride];
  float comb[Cfg::kGroups][G][kHeadDim];
  float comb_m[Cfg::kGroups][G];
  float comb_l[Cfg::kGroups][G];
  Piece pinfo[2];
  int stage_valid[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t qfull[2];
  uint64_t qempty[2];
  int abort_flag;
  int is_last;
  int wait_ok[Cfg::kCW];
  int end_flag[Cfg::kCW];
};

// Debug-only phase trace (build with -DPKV_TRACE=1): %globaltimer stamps of
// each CTA's phases, read back with pkv_debug_trace().
#ifndef PKV_TRACE
#define PKV_TRACE 0
#endif
#if PKV_TRACE
constexpr int kTraceCtas = 1024, kTraceEvents = 12;
__device__ unsigned long long g_trace[kTraceCtas][kTraceEvents];
#define TRACE(ev) do { if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x][ev] = global_timer_ns(); } while (0)
#define TRACE_ADD(ev, v) do { if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x][ev] += (v); } while (0)
#define TRACE_NOW() global_timer_ns()
#else
#define TRACE(ev) do { } while (0)
#define TRACE_ADD(ev, v) do { } while (0)
#define TRACE_NOW() 0ull
#endif

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
__device__ __forceinline__ long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Consumer: one 16-token block for one warp.
// ---------------------------------------------------------------------------
template <int G, int kPStride>
struct BlockMath {  // G = query heads this warp holds
  static constexpr bool kEven = (G % 2) == 0;
  static constexpr int F = kEven ? G / 2 : G;  // scores a lane owns after the scatter

  // Logical head held in register slot hs of a lane (see the reduce-scatter).
  __device__ static __forceinline__ int head_of_slot(int hs, int b0) {
    if constexpr (kEven) {
      int h = hs + b0 * (G / 2);
      return h >= G ? h - G : h;
    } else {
      return hs;
    }
  }

  __device__ static __forceinline__ void run(const uint8_t* stage, int nvalid, int lane,
                                             const float2 (&qf)[G][4], float (&m)[G],
                                             float (&lsum)[F], float2 (&acc)[G][4],
                                             float2 (*pbuf)[kPStride]) {
    const int half = lane >> 4;
    const int c = lane & 15;
    const int x = (lane >> 1) & 7;
    const int b0 = lane & 1;
    const uint8_t* Kt = stage;
    const uint8_t* Vt = stage + kTileBytes;

    // ---- partial scores over this lane's 8 dims, slot tt*G + hs ------------
    // Register slot tt of lane L holds token tt ^ x(L).  Across lane masks
    // 8/4/2 the partner lane holds the matching tokens in the upper half of
    // its slots, so each reduce-scatter step keeps the lower half and adds
    // the partner's upper half: no selects.  The first step (mask 8) is fused
    // into the loop so that only 4*G partial scores are live at a time.
    float sc[4 * G];
    #pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const int tok_lo = half * 8 + (tt ^ x);
      const int tok_hi = half * 8 + ((tt + 4) ^ x);
      const uint4 wl = lds128(Kt + tok_lo * (kHeadDim * 2) + c * 16);
      const uint4 wh = lds128(Kt + tok_hi * (kHeadDim * 2) + c * 16);
      const float2 l0 = bf16x2_to_float2(wl.x), l1 = bf16x2_to_float2(wl.y);
      const float2 l2 = bf16x2_to_float2(wl.z), l3 = bf16x2_to_float2(wl.w);
      const float2 h0 = bf16x2_to_float2(wh.x), h1 = bf16x2_to_float2(wh.y);
      const float2 h2 = bf16x2_to_float2(wh.z), h3 = bf16x2_to_float2(wh.w);
      #pragma unroll
      for (int hs = 0; hs < G; ++hs) {
        float2 a = fmul2(qf[hs][0], l0);
        a = ffma2(qf[hs][1], l1, a);
        a = ffma2(qf[hs][2], l2, a);
        a = ffma2(qf[hs][3], l3, a);
        float2 b = fmul2(qf[hs][0], h0);
        b = ffma2(qf[hs][1], h1, b);
        b = ffma2(qf[hs][2], h2, b);
        b = ffma2(qf[hs][3], h3, b);
        sc[tt * G + hs] = (a.x + a.y) + __shfl_xor_sync(0xffffffffu, b.x + b.y, 8);
      }
    }
    // ---- rest of the reduce-scatter across the 16 lanes of the half-warp --
    #pragma unroll
    for (int j = 0; j < 2 * G; ++j) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j + 2 * G], 4);
    #pragma unroll
    for (int j = 0; j < G; ++j) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j + G], 2);
    if constexpr (kEven) {
      #pragma unroll
      for (int j = 0; j < G / 2; ++j) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j + G / 2], 1);
    } else {
      #pragma unroll
      for (int j = 0; j < G; ++j) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j], 1);
    }
    // Now sc[j], j < F, is the full score of token tl = half*8 + x and
    // logical head head_of_slot(j, b0), already in the log2 domain.
    const int tl = half * 8 + x;
    const bool tok_ok = tl < nvalid;
    float bm[F];
    #pragma unroll
    for (int j = 0; j < F; ++j) {
      sc[j] = tok_ok ? sc[j] : -INFINITY;  // masked / unowned keys never count
      bm[j] = sc[j];
    }
    #pragma unroll
    for (int mask = 2; mask <= 16; mask <<= 1) {
      #pragma unroll
      for (int j = 0; j < F; ++j) bm[j] = fmaxf(bm[j], __shfl_xor_sync(0xffffffffu, bm[j], mask));
    }
    // Block maximum of every logical head, new running max and rescale factors.
    float mnew[G], alpha[G];
    if constexpr (kEven) {
      #pragma unroll
      for (int j = 0; j < F; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, bm[j], 1);
        const float lo = b0 ? other : bm[j];  // head j
        const float hi = b0 ? bm[j] : other;  // head j + G/2
        mnew[j] = fmaxf(m[j], lo);
        mnew[j + F] = fmaxf(m[j + F], hi);
      }
    } else {
      #pragma unroll
      for (int j = 0; j < G; ++j) mnew[j] = fmaxf(m[j], bm[j]);
    }
    bool changed = false;
    #pragma unroll
    for (int h = 0; h < G; ++h) {
      alpha[h] = fast_exp2(m[h] - mnew[h]);
      changed |= (mnew[h] != m[h]);
      m[h] = mnew[h];
    }
    // Probabilities of the owned scores; the lane's share of the normaliser.
    #pragma unroll
    for (int j = 0; j < F; ++j) {
      const int h = head_of_slot(j, b0);
      float mh, ah;
      if constexpr (kEven) {
        mh = b0 ? mnew[j + F] : mnew[j];
        ah = b0 ? alpha[j + F] : alpha[j];
      } else {
        mh = mnew[j];
        ah = alpha[j];
      }
      const float pj = fast_exp2(sc[j] - mh);
      lsum[j] = lsum[j] * ah + pj;
#if PKV_P_DUP
      if (kEven || b0 == 0) pbuf[tl][h] = make_float2(pj, pj);
#else
      if (kEven || b0 == 0) reinterpret_cast<float*>(pbuf[tl])[h] = pj;
#endif
    }
    __syncwarp();
    if (__any_sync(0xffffffffu, changed)) {
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        const float2 a2 = make_float2(alpha[h], alpha[h]);
        #pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][i] = fmul2(acc[h][i], a2);
      }
    }
    // ---- PV over this half's 8 tokens --------------------------------------
    #pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
      const int tok = half * 8 + tt;
      if (tok < nvalid) {
        const uint4 w = lds128(Vt + tok * (kHeadDim * 2) + c * 16);
        const float2 v0 = bf16x2_to_float2(w.x), v1 = bf16x2_to_float2(w.y);
        const float2 v2 = bf16x2_to_float2(w.z), v3 = bf16x2_to_float2(w.w);
#if PKV_P_DUP
        float2 pr[kPStride];
        #pragma unroll
        for (int i = 0; i < kPStride; i += 2) {
          const float4 t4 = *reinterpret_cast<const float4*>(&pbuf[tok][i]);
          pr[i] = make_float2(t4.x, t4.y);
          pr[i + 1] = make_float2(t4.z, t4.w);
        }
#else
        float prs[2 * kPStride];
        #pragma unroll
        for (int i = 0; i < 2 * kPStride; i += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(pbuf[tok]) + i);
          prs[i] = t4.x; prs[i + 1] = t4.y; prs[i + 2] = t4.z; prs[i + 3] = t4.w;
        }
#endif
        #pragma unroll
        for (int h = 0; h < G; ++h) {
#if PKV_P_DUP
          const float2 p2 = pr[h];
#else
          const float2 p2 = make_float2(prs[h], prs[h]);
#endif
          acc[h][0] = ffma2(p2, v0, acc[h][0]);
          acc[h][1] = ffma2(p2, v1, acc[h][1]);
          acc[h][2] = ffma2(p2, v2, acc[h][2]);
          acc[h][3] = ffma2(p2, v3, acc[h][3]);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// The plan.
// ---------------------------------------------------------------------------
// Sum over x = 1..n of ceil(x / 16): with n = 16m + t, 8m(m+1) + t(m+1).
__device__ __forceinline__ long long ceil16_prefix(long long n) {
  if (n <= 0) return 0;
  const long long m = n / kBlockSize, t = n % kBlockSize;
  return 8 * m * (m + 1) + t * (m + 1);
}

struct ReqInfo {
  int q0, qr, L;
  bool decode;  // has rows this kernel serves
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
  return ri;
}

// Blocks of rows 0..i-1 of a request (one KV head): row i sees L - qr + i + 1
// keys, i.e. ceil((L - qr + 1 + i) / 16) blocks.
__device__ __forceinline__ long long rows_blocks(const ReqInfo& ri, int i) {
  const long long a = (long long)ri.L - ri.qr + 1;
  return ceil16_prefix(a + i - 1) - ceil16_prefix(a - 1);
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(DecodeCfg<G>::kThreads) __maxnreg__(DecodeCfg<G>::kMaxRegs)
    decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecodeSmem<G>& sm = *reinterpret_cast<DecodeSmem<G>*>(smem_raw);
  volatile int* abort_flag = &sm.abort_flag;
  constexpr int kStages = DecodeSmem<G>::kStages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.num_reqs, Hkv = p.num_kv_heads;

  if (tid == 0) TRACE(0);
  if (tid == 0) {
    #pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], DecodeCfg<G>::kHS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.qfull[b], 1);
      mbar_init(&sm.qempty[b], DecodeCfg<G>::kCW);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Everything above overlaps the previous kernel's tail; every input may be
  // that kernel's output, so all reads come after this point.
  grid_dependency_wait();
  allow_dependent_launch();
  if (tid == 0) TRACE(1);

  if (warp == DecodeCfg<G>::kCW) {
    // ======================= producer warp =================================
    // Warm L2 with the part of the block table this CTA will probably read
    // (its share of the step if every row were full), while the plan loads.
    if (p.prefetch) {
      const long long entries = (long long)R * p.max_blocks;
      const long long est = entries * blockIdx.x / gridDim.x;
      const long long line0 = (est * 4) / 128 - 2;
      const long long lines = (entries * 4 + 127) / 128;
      const long long line = line0 + lane;
      if (line >= 0 && line < lines)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.block_tables) +
                                                     line * 128));
    }
    // ---- plan, pass 1: total blocks W of the decode rows (all KV heads) ----
    long long mine = 0;
    int nb_min = INT_MAX, nb_max = 0;
    for (int r = lane; r < R; r += 32) {
      const ReqInfo ri = load_request(p, r);
      if (ri.decode) {
        mine += rows_blocks(ri, ri.qr) * Hkv;
        nb_min = min(nb_min, ceil_div(ri.L - ri.qr + 1, kBlockSize));
        nb_max = max(nb_max, ceil_div(ri.L, kBlockSize));
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
    long long chunk = max((long long)p.min_chunk, ceil_div_ll(W, gridDim.x));
    if (p.align && nb_min == nb_max && W > 0) {
      // Uniform row-groups: cut each into equal pieces, or keep whole groups
      // together, so that piece boundaries coincide with CTA boundaries.
      const long long nb = nb_max;
      chunk = chunk < nb ? ceil_div_ll(nb, nb / chunk) : ceil_div_ll(chunk, nb) * nb;
    }
    const long long lo = (long long)blockIdx.x * chunk;
    const long long hi = min(W, lo + chunk);
    if (lane == 0) TRACE(2);

    const uint64_t pol = l2_policy_evict_first();
    uint32_t n = 0;  // CTA-wide block sequence number
    int j = 0;       // CTA-local piece index
    if (lo < hi) {
      // ---- pass 2: the request holding block lo, and where it starts -------
      int r = -1;
      long long pos = 0, base = 0;
      for (int b = 0; b < R; b += 32) {
        const int rr = b + lane;
        long long w = 0;
        if (rr < R) {
          const ReqInfo ri = load_request(p, rr);
          if (ri.decode) w = rows_blocks(ri, ri.qr) * Hkv;
        }
        long long incl = w;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const long long excl = incl - w;
        const unsigned own = __ballot_sync(0xffffffffu, w > 0 && base + excl <= lo && lo < base + incl);
        if (own) {
          const int src = __ffs(own) - 1;
          r = b + src;
          pos = base + __shfl_sync(0xffffffffu, excl, src);
          break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      // Walk the row-groups that intersect [lo, hi).
      if (r < 0) {
        record_error(p.err, kErrBounds);  // unreachable when the lengths are stable
        r = R;
      }
      ReqInfo ri = load_request(p, r < R ? r : 0);
      int i = 0;
      {  // first row of request r whose groups reach lo (binary search)
        int a = 0, b = ri.qr - 1;
        while (a < b) {
          const int mid = (a + b + 1) / 2;
          if (pos + rows_blocks(ri, mid) * Hkv <= lo) a = mid; else b = mid - 1;
        }
        i = a;
      }
      long long g = r < R ? pos + rows_blocks(ri, i) * Hkv : hi;  // start of row i, head 0
      int nb = ceil_div(ri.L - ri.qr + i + 1, kBlockSize);
      int k = (int)((lo - g) / nb);
      g += (long long)k * nb;
      while (g < hi && !*abort_flag) {
        // ---- one piece: row-group (r, i, k) = global blocks [g, g + nb) ----
        const long long s0 = max(g, lo), s1 = min(g + nb, hi);
        const long long c0 = g / chunk, c1 = (g + nb - 1) / chunk;
        Piece pc;
        pc.row = ri.q0 + i;
        pc.k = k;
        pc.b0 = (int)(s0 - g);
        pc.nblk = (int)(s1 - s0);
        pc.limit = ri.L - ri.qr + i + 1;
        pc.S = (int)(c1 - c0 + 1);
        pc.c0 = (int)c0;
        pc.odd0 = g != c0 * chunk;
        pc.slot = 2 * (int)blockIdx.x + (s0 == lo ? 0 : 1);
        const int ub = j & 1;
        if (j >= 2 && !mbar_wait(&sm.qempty[ub], ((j >> 1) - 1) & 1, p.err, abort_flag)) break;
        if (lane == 0) {
          sm.pinfo[ub] = pc;
          mbar_arrive_expect_tx(&sm.qfull[ub], G * kHeadDim * 2);
          bulk_copy_g2s(sm.qbuf[ub],
                        p.q + ((long long)pc.row * p.num_q_heads + (long long)k * G) * kHeadDim,
                        G * kHeadDim * 2, &sm.qfull[ub]);
        }
        const int32_t* bt = p.block_tables + (long long)r * p.max_blocks + pc.b0;
        for (int bb = 0; bb < pc.nblk && !*abort_flag; bb += 32) {
          const int cnt = min(32, pc.nblk - bb);
          const int ent = lane < cnt ? __ldg(bt + bb + lane) : 0;
          for (int xb = 0; xb < cnt; ++xb, ++n) {
            int phys = __shfl_sync(0xffffffffu, ent, xb);
            const int st = n % kStages;
            [[maybe_unused]] const unsigned long long tw0 = TRACE_NOW();
            if (n >= kStages &&
                !mbar_wait(&sm.empty[st], ((n / kStages) - 1) & 1, p.err, abort_flag))
              break;
            if (lane == 0) TRACE_ADD(8, TRACE_NOW() - tw0);
            if (lane == 0) {
              const bool valid = (unsigned)phys < (unsigned)p.num_blocks;
              if (!valid) {
                record_error(p.err, kErrBounds);
                phys = 0;
              }
              sm.stage_valid[st] = valid;
              const long long tile = ((long long)phys * Hkv + k) * (kTileBytes / 2);
              mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
              bulk_copy_g2s(sm.ring[st], p.k_pool + tile, kTileBytes, &sm.full[st], pol);
              bulk_copy_g2s(sm.ring[st] + kTileBytes, p.v_pool + tile, kTileBytes, &sm.full[st],
                            pol);
            }
            __syncwarp();
          }
        }
        ++j;
        // ---- advance to the next row-group ---------------------------------
        g += nb;
        if (++k == Hkv) {
          k = 0;
          if (++i == ri.qr) {
            i = 0;
            do {
              ++r;
              if (r >= R) break;
              ri = load_request(p, r);
            } while (!ri.decode);
            if (r >= R) break;
          }
          nb = ceil_div(ri.L - ri.qr + i + 1, kBlockSize);
        }
      }
    }
    // End marker: no more pieces for this CTA.
    const int ub = j & 1;
    if (j < 2 || mbar_wait(&sm.qempty[ub], ((j >> 1) - 1) & 1, p.err, abort_flag)) {
      if (lane == 0) {
        sm.pinfo[ub].row = kEndRow;
        mbar_arrive(&sm.qfull[ub]);
      }
    }
    return;
  }

  // ========================= consumer warps ================================
  using Cfg = DecodeCfg<G>;
  constexpr int GH = Cfg::kGH;  // heads of this warp: ho .. ho + GH - 1
  using BM = BlockMath<GH, DecodeSmem<G>::kPStride>;
  constexpr int F = BM::F;
  constexpr int kConsumerThreads = Cfg::kCW * 32;
  const int cw = warp;
  constexpr int kGroups = Cfg::kGroups;
  const int grp = cw / Cfg::kHS;       // the warp group that takes a block
  const int ho = (cw % Cfg::kHS) * GH;  // first head of this warp
  const int ct = tid;  // 0..127: the output dim this thread writes in the epilogue
  const int c = lane & 15;
  const int b0bit = lane & 1;
  uint32_t n_base = 0;
  for (int j = 0;; ++j) {
    const int ub = j & 1;
    const bool have_q = mbar_wait(&sm.qfull[ub], (j >> 1) & 1, p.err, abort_flag);
    Piece pc = sm.pinfo[ub];
    const bool is_end = !have_q || pc.row == kEndRow;
    // Range checks make every later index safe even after an abort.
    const bool in_range = !is_end && pc.row >= 0 && pc.row < p.num_q_tokens && pc.k >= 0 &&
                          pc.k < Hkv && pc.nblk >= 1 && pc.nblk <= p.max_blocks &&
                          pc.b0 >= 0 && pc.S >= 1 && pc.c0 >= 0 &&
                          2 * (pc.c0 + pc.S) <= p.num_slots && pc.slot >= 0 &&
                          pc.slot < p.num_slots;
    if (!in_range) pc.nblk = 0;
    float2 qf[GH][4];
    #pragma unroll
    for (int hs = 0; hs < GH; ++hs) {
      const int hl = ho + BM::head_of_slot(hs, b0bit);
      const uint4 w = lds128(&sm.qbuf[ub][hl * kHeadDim + c * 8]);
      const float2 s2 = make_float2(p.scale_log2, p.scale_log2);
      qf[hs][0] = fmul2(bf16x2_to_float2(w.x), s2);
      qf[hs][1] = fmul2(bf16x2_to_float2(w.y), s2);
      qf[hs][2] = fmul2(bf16x2_to_float2(w.z), s2);
      qf[hs][3] = fmul2(bf16x2_to_float2(w.w), s2);
    }
    __syncwarp();
    if (lane == 0 && !is_end) mbar_arrive(&sm.qempty[ub]);

    float m[GH], lsum[F];
    float2 acc[GH][4];
    #pragma unroll
    for (int h = 0; h < GH; ++h) {
      m[h] = kNegBig;
      #pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = make_float2(0.f, 0.f);
    }
    #pragma unroll
    for (int jj = 0; jj < F; ++jj) lsum[jj] = 0.f;

    for (int bi = (int)((grp + kGroups - n_base % kGroups) % kGroups); bi < pc.nblk;
         bi += kGroups) {
      const uint32_t n = n_base + bi;
      const int st = n % kStages;
      [[maybe_unused]] const unsigned long long tw0 = TRACE_NOW();
      const bool arrived = mbar_wait(&sm.full[st], (n / kStages) & 1, p.err, abort_flag);
      [[maybe_unused]] const unsigned long long tw1 = TRACE_NOW();
      if (n == 0 && lane == 0) TRACE(4);
      if (cw == 0 && lane == 0) TRACE_ADD(9, tw1 - tw0);
      const int first = (pc.b0 + bi) * kBlockSize;
      const int nvalid = (arrived && sm.stage_valid[st]) ? min(kBlockSize, pc.limit - first) : 0;
      BM::run(sm.ring[st], nvalid, lane, qf, m, lsum, acc, sm.pbuf[cw]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
      if (cw == 0 && lane == 0) {
        TRACE_ADD(10, TRACE_NOW() - tw1);
        TRACE_ADD(11, 1);
      }
    }
    n_base += pc.nblk;
    if (ct == 0 && !is_end) TRACE(5);

    // ---- combine the four warp groups' states -----------------------------
    if (is_end) {
      // The end marker carries no work: only agree on it, then leave.
      if (lane == 0) {
        sm.wait_ok[cw] = 0;
        sm.end_flag[cw] = 1;
      }
      named_barrier(1, kConsumerThreads);
      break;
    }
    float lall[GH];
    {
      float l2[F];
      #pragma unroll
      for (int jj = 0; jj < F; ++jj) {
        l2[jj] = lsum[jj];
        #pragma unroll
        for (int mask = 2; mask <= 16; mask <<= 1)
          l2[jj] += __shfl_xor_sync(0xffffffffu, l2[jj], mask);
      }
      if constexpr (BM::kEven) {
        #pragma unroll
        for (int jj = 0; jj < F; ++jj) {
          const float other = __shfl_xor_sync(0xffffffffu, l2[jj], 1);
          lall[jj] = b0bit ? other : l2[jj];
          lall[jj + F] = b0bit ? l2[jj] : other;
        }
      } else {
        #pragma unroll
        for (int jj = 0; jj < GH; ++jj) lall[jj] = l2[jj];
      }
    }
    #pragma unroll
    for (int h = 0; h < GH; ++h)
      #pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[h][i].x += __shfl_xor_sync(0xffffffffu, acc[h][i].x, 16);
        acc[h][i].y += __shfl_xor_sync(0xffffffffu, acc[h][i].y, 16);
      }
    if (lane < 16) {
      #pragma unroll
      for (int h = 0; h < GH; ++h) {
        float4* dst = reinterpret_cast<float4*>(&sm.comb[grp][ho + h][c * 8]);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
    }
    if (lane == 0) {
      #pragma unroll
      for (int h = 0; h < GH; ++h) {
        sm.comb_m[grp][ho + h] = m[h];
        sm.comb_l[grp][ho + h] = lall[h];
      }
      sm.wait_ok[cw] = in_range;
      sm.end_flag[cw] = is_end;
    }
    named_barrier(1, kConsumerThreads);

    // When every warp's wait succeeded, all four hold the same piece (it
    // cannot change before all four have released the q buffer), so `ok` and
    // `end` are uniform across the consumer warps and so are the barriers.
    bool ok = true, end = false;
    #pragma unroll
    for (int w = 0; w < Cfg::kCW; ++w) {
      ok = ok && sm.wait_ok[w];
      end = end || sm.end_flag[w];
    }
    if (end) break;  // another warp saw the end marker (only after an abort)
    // Epilogue: the consumer threads stride over the g x 128 outputs.
    const long long out_row = ((long long)pc.row * p.num_q_heads + (long long)pc.k * G) * kHeadDim;
    #pragma unroll 1
    for (int idx = ct; idx < G * kHeadDim; idx += kConsumerThreads) {
      const int h = idx / kHeadDim, d = idx % kHeadDim;
      float M = sm.comb_m[0][h];
      #pragma unroll
      for (int w = 1; w < kGroups; ++w) M = fmaxf(M, sm.comb_m[w][h]);
      float num = 0.f, den = 0.f;
      #pragma unroll
      for (int w = 0; w < kGroups; ++w) {
        const float e = fast_exp2(sm.comb_m[w][h] - M);
        num += e * sm.comb[w][h][d];
        den += e * sm.comb_l[w][h];
      }
      const float res = den > 0.f ? num / den : 0.f;
      if (ok && pc.S > 1) {
        const long long slot = (long long)pc.slot * G + h;
        p.ws_o[slot * kHeadDim + d] = res;
        if (d == 0) *reinterpret_cast<float2*>(p.ws_ml + slot * 2) = make_float2(M, den);
      } else if (ok) {
        p.out[out_row + h * kHeadDim + d] = __float2bfloat16_rn(res);
      }
    }
    if (ok && pc.S > 1) {
      // Ticket: the barrier orders every thread's partial stores before
      // thread 0's fence, whose release is cumulative, then the atomic.  The
      // piece that draws the last ticket fences again (acquire) and merges.
      named_barrier(1, kConsumerThreads);
      if (ct == 0) {
        __threadfence();
        int* cnt = p.ws_cnt + (long long)pc.row * Hkv + pc.k;
        const int old = atomicAdd(cnt, 1);
        const int last = (old == pc.S - 1);
        if (last) {
          *cnt = 0;  // every piece has arrived: leave the counter at zero
          __threadfence();
        }
        sm.is_last = last;
      }
      named_barrier(1, kConsumerThreads);
      if (sm.is_last) {
        // Log-sum-exp merge of the row-group's pieces, in piece order, one
        // pass with a running maximum; loads of four pieces are in flight at
        // once.
        #pragma unroll 1
        for (int idx = ct; idx < G * kHeadDim; idx += kConsumerThreads) {
          const int h = idx / kHeadDim, d = idx % kHeadDim;
          float M = kNegBig, num = 0.f, den = 0.f;
          #pragma unroll 4
          for (int s = 0; s < pc.S; ++s) {
            const int slot = 2 * (pc.c0 + s) + ((s == 0 && pc.odd0) ? 1 : 0);
            const long long sl = (long long)slot * G + h;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + sl * 2));
            const float o = __ldcg(p.ws_o + sl * kHeadDim + d);
            const float Mn = fmaxf(M, ml.x);
            const float a = fast_exp2(M - Mn), w = fast_exp2(ml.x - Mn) * ml.y;
            num = num * a + w * o;
            den = den * a + w;
            M = Mn;
          }
          p.out[out_row + h * kHeadDim + d] = __float2bfloat16_rn(num / den);
        }
      }
    }
    // Close the piece: nobody rewrites comb/is_last before everyone is done.
    named_barrier(1, kConsumerThreads);
    if (ct == 0 && !end) TRACE(6);
    if (end) break;
  }
  if (ct == 0) TRACE(7);
}

template <int G>
cudaError_t launch_decode_g(const DecodeParams& p, int grid, cudaStream_t stream) {
  if (getenv("PKV_DEBUG")) {
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<G>, DecodeCfg<G>::kThreads,
                                                  sizeof(DecodeSmem<G>));
    fprintf(stderr, "decode_kernel<%d>: smem %zu B, %d CTAs/SM resident, grid %d\n", G,
            sizeof(DecodeSmem<G>), occ, grid);
  }
  const size_t smem = sizeof(DecodeSmem<G>);
  static unsigned long long configured = 0;  // bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    // Two CTAs per SM need the largest shared-memory carveout.
    e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(DecodeCfg<G>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel<G>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

#if PKV_TRACE
cudaError_t decode_trace(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace));
}
#endif

int decode_ctas_per_sm(int group) {
  switch (group) {
    case 1: return DecodeCfg<1>::kMinCtas;
    case 2: return DecodeCfg<2>::kMinCtas;
    case 3: return DecodeCfg<3>::kMinCtas;
    case 4: return DecodeCfg<4>::kMinCtas;
    case 5: return DecodeCfg<5>::kMinCtas;
    case 6: return DecodeCfg<6>::kMinCtas;
    case 7: return DecodeCfg<7>::kMinCtas;
    default: return DecodeCfg<8>::kMinCtas;
  }
}

int decode_grid(int sm_count, int group) { return sm_count * decode_ctas_per_sm(group); }

WorkspaceLayout decode_workspace_layout(int num_q_tokens, int num_kv_heads, int group,
                                        int sm_count) {
  WorkspaceLayout w;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  w.num_slots = 2 * sm_count * 2;  // two partial pieces per CTA, up to two CTAs per SM
  w.cnt_off = 0;
  w.ml_off = up((size_t)num_q_tokens * num_kv_heads * sizeof(int));
  w.o_off = w.ml_off + up((size_t)w.num_slots * group * 2 * sizeof(float));
  w.total = w.o_off + up((size_t)w.num_slots * group * kHeadDim * sizeof(float));
  return w;
}

cudaError_t launch_decode(const DecodeParams& p, int group, int grid, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_g<1>(p, grid, stream);
    case 2: return launch_decode_g<2>(p, grid, stream);
    case 3: return launch_decode_g<3>(p, grid, stream);
    case 4: return launch_decode_g<4>(p, grid, stream);
    case 5: return launch_decode_g<5>(p, grid, stream);
    case 6: return launch_decode_g<6>(p, grid, stream);
    case 7: return launch_decode_g<7>(p, grid, stream);
    case 8: return launch_decode_g<8>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
