// pkv_decode_kernel.cuh -- paged decode attention with split context and a
// fused log-sum-exp merge, for sm_103a, over bf16 or e4m3 pools.  Included by
// pkv_decode.cu (bf16 pools) and pkv_decode_fp8.cu (e4m3 pools), which
// compile in parallel.
//
// What it computes (per query row t of request r, KV head k, and the g query
// heads h = k*g .. k*g+g-1 that share KV head k): the softmax-weighted sum of
// V over the keys the row may see, gathered block by block through the
// request's block table (The Serving Playbook, "The block table lives in the
// hottest kernel in the system").
//
// How, on GB300:
//  * One CTA serves all g query heads of a KV head, so each (block, KV head)
//    tile -- 4 KiB of K and 4 KiB of V, contiguous in the pool (2 KiB each
//    for an e4m3 pool) -- leaves HBM once per row.
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
//  * e4m3 pools (The Serving Playbook, "Quantized serving"): a code stands
//    for decode(code) * scale[KV head].  The key scale
//    is folded into q with scale*log2(e), the value scale multiplies the
//    normalised output; codes widen to fp32 through the hardware
//    e4m3x2 -> f16x2 conversion.
#pragma once
#include <climits>
#include <cstdio>
#include <cstdlib>

#include <cuda_fp8.h>

#include "pkv_internal.h"
#include "pkv_plan.cuh"

namespace pkv {
namespace {

// Element type of the pools: the tile of one (block, KV head) and how a
// lane widens its 8 consecutive elements of one token row to fp32.
struct KvBf16 {
  static constexpr int kTileBytes = kBlockSize * kHeadDim * 2;  // 4 KiB
  static constexpr int kRowBytes = kHeadDim * 2;
  static constexpr bool kFp8 = false;
  __device__ static __forceinline__ void load8(const uint8_t* row, int c, float2 (&v)[4]) {
    const uint4 w = lds128(row + c * 16);
    v[0] = bf16x2_to_float2(w.x);
    v[1] = bf16x2_to_float2(w.y);
    v[2] = bf16x2_to_float2(w.z);
    v[3] = bf16x2_to_float2(w.w);
  }
};
struct KvE4m3 {
  static constexpr int kTileBytes = kBlockSize * kHeadDim;  // 2 KiB
  static constexpr int kRowBytes = kHeadDim;
  static constexpr bool kFp8 = true;
  __device__ static __forceinline__ void load8(const uint8_t* row, int c, float2 (&v)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + c * 8);
    v[0] = e4m3x2_to_float2(w.x & 0xffffu);
    v[1] = e4m3x2_to_float2(w.x >> 16);
    v[2] = e4m3x2_to_float2(w.y & 0xffffu);
    v[3] = e4m3x2_to_float2(w.y >> 16);
  }
};

// Warp layout: blocks are consumed by four warp groups of one warp each, in
// turn; a warp holds all g heads of the group.
template <int G>
struct DecodeCfg {
  static constexpr int kGH = G;                                   // heads per warp
  static constexpr int kMinCtas = (kGH <= 6) ? 2 : 1;             // CTAs per SM
  static constexpr int kGroups = 4;                               // consumer warp groups
  static constexpr int kCW = kGroups;                             // consumer warps
  static constexpr int kThreads = (kCW + 1) * 32;                 // + producer warp
  // Registers per thread that still let kMinCtas CTAs share an SM: each of
  // the four SM sub-partitions owns a quarter of the register file (16384)
  // and holds every fourth resident warp.
  static constexpr int kWarpsSm = kMinCtas * (kCW + 1);
  static constexpr int kRegFit = (16384 / (32 * ((kWarpsSm + 3) / 4))) / 8 * 8;
  static constexpr int kMaxRegs = kRegFit > 255 ? 255 : kRegFit;
};

// Ring depth: about 64 KiB of stages per CTA when two CTAs share an SM
// (8 bf16 tiles pairs, 16 e4m3 ones), about 160 KiB when one CTA has the SM
// to itself, rounded up to a multiple of the warp-group count.  The rounding
// is a correctness condition, not a tuning choice: a consumer waits on a
// stage's full barrier by phase parity, which is only unambiguous if the
// stage's previous phase (block n - stages) was consumed by the same warp
// group, i.e. if the group count divides the ring depth.  Otherwise a warp
// can run two phases ahead, pass a stale parity and read a stage that is
// still being filled.
template <int G, class KV>
constexpr int stages_for() {
  constexpr int kWant =
      (DecodeCfg<G>::kMinCtas == 2 ? 8 : 20) * (KvBf16::kTileBytes / KV::kTileBytes);
  constexpr int kGroups = DecodeCfg<G>::kGroups;
  return (kWant + kGroups - 1) / kGroups * kGroups;
}
constexpr float kNegBig = -1.0e30f;          // "no key seen yet" running max
constexpr float kLazyMargin = 8.f;           // log2 of the largest probability allowed
using plan::Piece;
using plan::kEndRow;


template <int G, class KV>
struct __align__(128) DecodeSmem {
  using Cfg = DecodeCfg<G>;
  static constexpr int kStages = stages_for<G, KV>();
  static_assert(kStages % Cfg::kGroups == 0, "each stage must stay with one warp group");
  static constexpr int kStageBytes = 2 * KV::kTileBytes;  // K tile then V tile
  // Probabilities of one block, stored twice ({p, p}) so that the PV loop
  // feeds packed fp32 FMAs straight from 16-byte loads.
  static constexpr int kPStride = ((Cfg::kGH + 3) & ~3) / 2;  // float2 slots = 2 floats each
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
  WaitCtl wait;                   // abort flag and wait limit of the bounded waits
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
template <int G, int kPStride, class KV>
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

  // acc += p(tok) * V[tok] for this lane's 8 dims and the warp's G heads.
  __device__ static __forceinline__ void pv_token(const uint8_t* Vt, int tok, int c,
                                                  float2 (&acc)[G][4],
                                                  float2 (*pbuf)[kPStride]) {
    float2 vv[4];
    KV::load8(Vt + tok * KV::kRowBytes, c, vv);
    float prs[2 * kPStride];
    #pragma unroll
    for (int i = 0; i < 2 * kPStride; i += 4) {
      const float4 t4 =
          *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(pbuf[tok]) + i);
      prs[i] = t4.x; prs[i + 1] = t4.y; prs[i + 2] = t4.z; prs[i + 3] = t4.w;
    }
    #pragma unroll
    for (int h = 0; h < G; ++h) {
      const float2 p2 = make_float2(prs[h], prs[h]);
      #pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = ffma2(p2, vv[i], acc[h][i]);
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
    const uint8_t* Vt = stage + KV::kTileBytes;

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
      float2 l[4], hv[4];
      KV::load8(Kt + tok_lo * KV::kRowBytes, c, l);
      KV::load8(Kt + tok_hi * KV::kRowBytes, c, hv);
      #pragma unroll
      for (int hs = 0; hs < G; ++hs) {
        float2 a = fmul2(qf[hs][0], l[0]);
        a = ffma2(qf[hs][1], l[1], a);
        a = ffma2(qf[hs][2], l[2], a);
        a = ffma2(qf[hs][3], l[3], a);
        float2 b = fmul2(qf[hs][0], hv[0]);
        b = ffma2(qf[hs][1], hv[1], b);
        b = ffma2(qf[hs][2], hv[2], b);
        b = ffma2(qf[hs][3], hv[3], b);
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
    // Running max of each owned score's head.  The probabilities of a block
    // are taken against the running max as it stands; it is raised (and the
    // state rescaled) only when some score of the block exceeds it by more
    // than kLazyMargin, so p stays <= 2^kLazyMargin and the common block
    // needs no cross-lane max reduction.  The result is the same softmax:
    // every term of the output and of the normaliser carries the same
    // factor 2^-m, whatever m is.
    float mo[F];
    bool over = false;
    #pragma unroll
    for (int j = 0; j < F; ++j) {
      sc[j] = tok_ok ? sc[j] : -INFINITY;  // masked / unowned keys never count
      if constexpr (kEven) mo[j] = b0 ? m[j + F] : m[j];
      else mo[j] = m[j];
      over |= sc[j] > mo[j] + kLazyMargin;
    }
    if (__any_sync(0xffffffffu, over)) {
      float bm[F];
      #pragma unroll
      for (int j = 0; j < F; ++j) bm[j] = sc[j];
      #pragma unroll
      for (int mask = 2; mask <= 16; mask <<= 1) {
        #pragma unroll
        for (int j = 0; j < F; ++j) bm[j] = fmaxf(bm[j], __shfl_xor_sync(0xffffffffu, bm[j], mask));
      }
      // Block maximum of every logical head, new running max, rescale factors.
      float mnew[G];
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
      float alpha[G];
      bool changed = false;
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        alpha[h] = fast_exp2(m[h] - mnew[h]);
        changed |= (mnew[h] != m[h]);
        m[h] = mnew[h];
      }
      #pragma unroll
      for (int j = 0; j < F; ++j) {
        if constexpr (kEven) {
          mo[j] = b0 ? mnew[j + F] : mnew[j];
          lsum[j] *= b0 ? alpha[j + F] : alpha[j];
        } else {
          mo[j] = mnew[j];
          lsum[j] *= alpha[j];
        }
      }
      if (__any_sync(0xffffffffu, changed)) {
        #pragma unroll
        for (int h = 0; h < G; ++h) {
          const float2 a2 = make_float2(alpha[h], alpha[h]);
          #pragma unroll
          for (int i = 0; i < 4; ++i) acc[h][i] = fmul2(acc[h][i], a2);
        }
      }
    }
    // Probabilities of the owned scores; the lane's share of the normaliser.
    #pragma unroll
    for (int j = 0; j < F; ++j) {
      const int h = head_of_slot(j, b0);
      const float pj = fast_exp2(sc[j] - mo[j]);
      lsum[j] += pj;
      if (kEven || b0 == 0) reinterpret_cast<float*>(pbuf[tl])[h] = pj;
    }
    __syncwarp();
    // ---- PV over this half's 8 tokens --------------------------------------
    // Full blocks (every block but a row's last) take a loop without
    // per-token checks.
    if (nvalid >= kBlockSize) {
      #pragma unroll
      for (int tt = 0; tt < 8; ++tt) pv_token(Vt, half * 8 + tt, c, acc, pbuf);
    } else {
      #pragma unroll
      for (int tt = 0; tt < 8; ++tt)
        if (half * 8 + tt < nvalid) pv_token(Vt, half * 8 + tt, c, acc, pbuf);
    }
  }
};

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int G, class KV>
__global__ void __launch_bounds__(DecodeCfg<G>::kThreads) __maxnreg__(DecodeCfg<G>::kMaxRegs)
    decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  using Smem = DecodeSmem<G, KV>;
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  WaitCtl* abort_flag = &sm.wait;
  constexpr int kStages = Smem::kStages;
  constexpr int kStageBytes = Smem::kStageBytes;
  constexpr int kTile = KV::kTileBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.num_kv_heads;

  if (tid == 0) TRACE(0);
  if (tid == 0) {
    #pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.qfull[b], 1);
      mbar_init(&sm.qempty[b], DecodeCfg<G>::kCW);
    }
    sm.wait.abort = 0;
    sm.wait.limit_ns = p.wait_limit_ns;
    fence_barrier_init();
  }
  __syncthreads();
  // Everything above overlaps the previous kernel's tail.  The consumers
  // wait for that kernel here; the producer first builds the plan, which
  // reads only seq_lens and query_start_loc (with early_plan set, the caller
  // guarantees the previous kernel does not write them), and waits before
  // its first read of q, the block table or the pools.  Every thread lets
  // the next kernel launch only after its own wait, so that kernel may rely
  // on everything before this one having completed.
  // With early_kv the previous kernel is the append of this step's new
  // tokens: before the wait the producer reads the lengths, the block table
  // and blocks without a new token, and waits before the first block holding
  // one (and before it blocks on the consumers).  If that append lets this
  // grid launch as soon as the append starts (early_q unset), q, out and the
  // workspace may still belong to the kernel before the append: Q copies are
  // then issued after the wait and the consumers wait before anything else.
  if (!p.early_kv && (warp != DecodeCfg<G>::kCW || !p.early_plan)) {
    grid_dependency_wait();
    allow_dependent_launch();
  }
  if (tid == 0) TRACE(1);

  if (warp == DecodeCfg<G>::kCW) {
    // ======================= producer warp =================================
    plan::Range rg;
    plan::Walker wk;
    plan::plan_cta(p, lane, rg, wk);
    if (lane == 0) TRACE(2);

    const uint64_t pol = l2_policy_evict_first();
    uint32_t n = 0;  // CTA-wide block sequence number
    int j = 0;       // CTA-local piece index
    bool waited = !p.early_kv;
    if (p.early_plan && !p.early_kv) {
      grid_dependency_wait();
      allow_dependent_launch();
    }
    // Q copies of pieces met before the wait (at most the two buffers'),
    // issued once it has been taken.
    int q_pend = 0;
    const __nv_bfloat16 *q_src0 = nullptr, *q_src1 = nullptr;
    auto take_wait = [&]() {
      if (!waited) {
        grid_dependency_wait();  // the append of this step's tokens is complete
        allow_dependent_launch();
        waited = true;
      }
      if (lane == 0 && (q_pend & 1)) bulk_copy_g2s(sm.qbuf[0], q_src0, G * kHeadDim * 2, &sm.qfull[0]);
      if (lane == 0 && (q_pend & 2)) bulk_copy_g2s(sm.qbuf[1], q_src1, G * kHeadDim * 2, &sm.qfull[1]);
      q_pend = 0;
    };
    Piece pc;
    while (!abort_flag->abort && wk.next(p, pc)) {
      // ---- one piece: blocks [b0, b0 + nblk) of row-group (row, k) --------
      const int k = pc.k;
      const int ub = j & 1;
      if (j >= 2) {
        if (!waited || q_pend) take_wait();
        if (!mbar_wait(&sm.qempty[ub], ((j >> 1) - 1) & 1, p.err, abort_flag)) break;
      }
      const __nv_bfloat16* qsrc =
          p.q + ((long long)pc.row * p.num_q_heads + (long long)k * G) * kHeadDim;
      if (lane == 0) {
        sm.pinfo[ub] = pc;
        mbar_arrive_expect_tx(&sm.qfull[ub], G * kHeadDim * 2);
        if (waited || p.early_q) bulk_copy_g2s(sm.qbuf[ub], qsrc, G * kHeadDim * 2, &sm.qfull[ub]);
      }
      if (!waited && !p.early_q) {
        q_pend |= 1 << ub;
        if (ub == 0) q_src0 = qsrc; else q_src1 = qsrc;
      }
      const int32_t* bt = p.block_tables + (long long)pc.r * p.max_blocks + pc.b0;
      for (int bb = 0; bb < pc.nblk && !abort_flag->abort; bb += 32) {
        const int cnt = min(32, pc.nblk - bb);
        const int ent = lane < cnt ? __ldg(bt + bb + lane) : 0;
        for (int xb = 0; xb < cnt; ++xb, ++n) {
          int phys = __shfl_sync(0xffffffffu, ent, xb);
          const int st = n % kStages;
          // Before blocking on the consumers, or before a block with a new token.
          if (n >= kStages || pc.b0 + bb + xb >= pc.fresh) {
            if (!waited || q_pend) take_wait();
          }
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
            const long long tile = ((long long)phys * Hkv + k) * kTile;
            mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
            bulk_copy_g2s(sm.ring[st], p.k_pool + tile, kTile, &sm.full[st], pol);
            bulk_copy_g2s(sm.ring[st] + kTile, p.v_pool + tile, kTile, &sm.full[st], pol);
          }
          __syncwarp();
        }
      }
      ++j;
    }
    // The CTA finishes after the previous kernel in any case; Q copies still
    // pending are issued unless the CTA is giving up.
    if (abort_flag->abort) q_pend = 0;
    take_wait();
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
  if (p.early_kv && !p.early_q) grid_dependency_wait();  // out and the workspace are written below
  using Cfg = DecodeCfg<G>;
  constexpr int GH = Cfg::kGH;  // heads of this warp: all G of the group
  using BM = BlockMath<GH, Smem::kPStride, KV>;
  constexpr int F = BM::F;
  constexpr int kConsumerThreads = Cfg::kCW * 32;
  const int cw = warp;
  constexpr int kGroups = Cfg::kGroups;
  const int grp = cw;  // the warp group (one warp) that takes a block
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
    // Per-KV-head dequantisation scales of an e4m3 pool: the key scale joins
    // the softmax scale in q, the value scale multiplies the output.
    float kscale = 1.f, vscale = 1.f;
    if constexpr (KV::kFp8) {
      if (in_range) {
        kscale = __ldg(p.k_scale + pc.k);
        vscale = __ldg(p.v_scale + pc.k);
      }
    }
    float2 qf[GH][4];
    #pragma unroll
    for (int hs = 0; hs < GH; ++hs) {
      const int hl = BM::head_of_slot(hs, b0bit);
      const uint4 w = lds128(&sm.qbuf[ub][hl * kHeadDim + c * 8]);
      const float qs = p.scale_log2 * kscale;
      const float2 s2 = make_float2(qs, qs);
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
        float4* dst = reinterpret_cast<float4*>(&sm.comb[grp][h][c * 8]);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
    }
    if (lane == 0) {
      #pragma unroll
      for (int h = 0; h < GH; ++h) {
        sm.comb_m[grp][h] = m[h];
        sm.comb_l[grp][h] = lall[h];
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
        p.out[out_row + h * kHeadDim + d] = __float2bfloat16_rn(res * vscale);
      }
    }
    if (ok && pc.S > 1) {
      // Ticket: the barrier orders every thread's partial stores before
      // thread 0's acquire-release atomic, whose release is cumulative; the
      // piece that draws the last ticket has acquired the others' and merges.
      named_barrier(1, kConsumerThreads);
      if (ct == 0) {
        int* cnt = p.ws_cnt + (long long)pc.row * Hkv + pc.k;
        const int old = atom_add_acq_rel_gpu(cnt, 1);
        const int last = (old == pc.S - 1);
        if (last) *cnt = 0;  // every piece has arrived: leave the counter at zero
        sm.is_last = last;
      }
      named_barrier(1, kConsumerThreads);
      if (sm.is_last) {
        // Log-sum-exp merge of the row-group's pieces, in piece order, one
        // pass with a running maximum; each piece's states of every head this
        // thread merges are loaded together (one L2 round trip per piece).
        static_assert(kConsumerThreads == kHeadDim, "one output dim per consumer thread");
        const int d = ct;
        float M[G], num[G], den[G];
        #pragma unroll
        for (int h = 0; h < G; ++h) {
          M[h] = kNegBig;
          num[h] = den[h] = 0.f;
        }
        #pragma unroll 1
        for (int s = 0; s < pc.S; ++s) {
          const int slot = 2 * (pc.c0 + s) + ((s == 0 && pc.odd0) ? 1 : 0);
          float2 ml[G];
          float o[G];
          #pragma unroll
          for (int h = 0; h < G; ++h) {
            const long long sl = (long long)slot * G + h;
            ml[h] = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + sl * 2));
            o[h] = __ldcg(p.ws_o + sl * kHeadDim + d);
          }
          #pragma unroll
          for (int h = 0; h < G; ++h) {
            const float Mn = fmaxf(M[h], ml[h].x);
            const float a = fast_exp2(M[h] - Mn), w = fast_exp2(ml[h].x - Mn) * ml[h].y;
            num[h] = num[h] * a + w * o[h];
            den[h] = den[h] * a + w;
            M[h] = Mn;
          }
        }
        #pragma unroll
        for (int h = 0; h < G; ++h)
          p.out[out_row + h * kHeadDim + d] = __float2bfloat16_rn(num[h] / den[h] * vscale);
      }
    }
    // Close the piece: nobody rewrites comb/is_last before everyone is done.
    named_barrier(1, kConsumerThreads);
    if (ct == 0 && !end) TRACE(6);
    if (end) break;
  }
  if (ct == 0) TRACE(7);
}

template <int G, class KV>
cudaError_t launch_decode_g(const DecodeParams& p, int grid, cudaStream_t stream) {
  using Smem = DecodeSmem<G, KV>;
  const size_t smem = sizeof(Smem);
  static unsigned long long configured = 0;  // bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(decode_kernel<G, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    // Two CTAs per SM need the largest shared-memory carveout.
    e = cudaFuncSetAttribute(decode_kernel<G, KV>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
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
  e = cudaLaunchKernelEx(&cfg, decode_kernel<G, KV>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace
}  // namespace pkv
