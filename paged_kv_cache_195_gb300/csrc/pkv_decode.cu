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
//  * Parallelism comes from the KV axis: each row's blocks are cut into
//    splits ("units") sized by a device-side plan from the step's lengths
//    (Flash-Decoding: The Serving Playbook, "Kernel fusion, briefly").  Each
//    CTA keeps an online-softmax state per split (running max, normaliser,
//    rescaled output: LLM 7 - Efficient LLM Serving, sec. 2 "Online Softmax
//    Makes Tiling Possible").  The last CTA to finish a row merges the splits
//    by log-sum-exp (the "second pass rescales the partials" step), found with
//    one atomic counter per row: no extra launch, deterministic merge order.
//  * A producer warp walks the CTA's units and issues cp.async.bulk copies of
//    whole tiles into an 8-stage shared-memory ring (mbarrier-tracked);
//    four consumer warps take ring stages round-robin.  The 16 KiB per tile
//    pair in flight per stage keeps ~128 KiB of loads outstanding per SM.
//  * Consumers: lane = (token half, 16-byte chunk of d).  q for all g heads of
//    the lane's chunk stays in registers; QK partial sums over the lane's 8
//    dims are reduced across the 16 lanes of a half-warp by a reduce-scatter
//    whose register order is permuted per lane so that no selects are needed;
//    softmax in fp32 (exp2 with scale*log2(e) folded into q); PV accumulates
//    in packed fp32 (fma.rn.f32x2).
//  * The plan (per-request unit counts and their prefix sum) is recomputed by
//    every CTA from seq_lens / query_start_loc in device memory, so the
//    launch shape depends only on bounds: the call is CUDA-graph capturable.
#include <climits>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 8;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr float kNegBig = -1.0e30f;          // "no key seen yet" running max

struct UnitInfo {
  int row;    // global query row
  int k;      // KV head
  int b0;     // first logical block
  int nblk;   // blocks in this unit (may be 0)
  int limit;  // keys visible to this row: positions < limit
  int S;      // splits of this (row, KV head)
  int unit;   // global unit id (workspace slot of this split)
  int base;   // workspace slot of split 0 of this row
};

template <int G>
struct __align__(128) DecodeSmem {
  static constexpr int kPStride = (G + 3) & ~3;
  uint8_t ring[kStages][kStageBytes];
  __nv_bfloat16 qbuf[2][G * kHeadDim];
  float pbuf[kConsumerWarps][kBlockSize][kPStride];
  float comb[kConsumerWarps][G][kHeadDim];
  float comb_m[kConsumerWarps][G];
  float comb_l[kConsumerWarps][G];
  UnitInfo uinfo[2];
  int stage_valid[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t qfull[2];
  uint64_t qempty[2];
  long long red[kDecodeThreads / 32];
  int total_units;
  int abort_flag;
  int stop;
  int is_last;
  int wait_ok[kConsumerWarps];
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Inclusive block-wide scan of one value per thread (all threads call).
template <typename T>
__device__ T block_inclusive_scan(T v, T* red, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  #pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) red[warp] = v;
  __syncthreads();
  T before = 0, all = 0;
  #pragma unroll
  for (int w = 0; w < kDecodeThreads / 32; ++w) {
    if (w < warp) before += red[w];
    all += red[w];
  }
  __syncthreads();
  *total = all;
  return v + before;
}

// ---------------------------------------------------------------------------
// Consumer: one 16-token block for one warp.
// ---------------------------------------------------------------------------
template <int G>
struct BlockMath {
  static constexpr bool kEven = (G % 2) == 0;
  static constexpr int F = kEven ? G / 2 : G;  // scores a lane owns after the scatter
  static constexpr int kPStride = DecodeSmem<G>::kPStride;

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
                                             float (*pbuf)[kPStride]) {
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
      if (kEven || b0 == 0) pbuf[tl][h] = pj;
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
        float pr[kPStride];
        #pragma unroll
        for (int i = 0; i < kPStride; i += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(&pbuf[tok][i]);
          pr[i] = t4.x; pr[i + 1] = t4.y; pr[i + 2] = t4.z; pr[i + 3] = t4.w;
        }
        #pragma unroll
        for (int h = 0; h < G; ++h) {
          const float2 p2 = make_float2(pr[h], pr[h]);
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
// The kernel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool request_ok(const DecodeParams& p, int q0, int q1, int L) {
  const int qr = q1 - q0;
  return q0 >= 0 && qr >= 0 && q1 <= p.num_q_tokens && qr <= L &&
         L <= p.max_blocks * kBlockSize;
}

// Work units of request r: its decode rows x KV heads x splits.
__device__ __forceinline__ long long request_units(const DecodeParams& p, int r, int chunk,
                                                   long long* work) {
  const int q0 = p.qsl[r], q1 = p.qsl[r + 1], L = p.seq_lens[r];
  const int qr = q1 - q0;
  if (!request_ok(p, q0, q1, L) || qr == 0 || qr >= p.prefill_min_q) {
    *work = 0;
    return 0;
  }
  const int nb = ceil_div(L, kBlockSize);
  *work = (long long)qr * nb;
  return chunk > 0 ? (long long)qr * p.num_kv_heads * ceil_div(nb, chunk) : 0;
}

template <int G>
__global__ void __launch_bounds__(kDecodeThreads, (G <= 6 ? 2 : 1))
    decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecodeSmem<G>& sm = *reinterpret_cast<DecodeSmem<G>*>(smem_raw);
  int* prefix = reinterpret_cast<int*>(smem_raw + sizeof(DecodeSmem<G>));  // [R+1]
  volatile int* abort_flag = &sm.abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.num_reqs, Hkv = p.num_kv_heads;

  if (tid == 0) {
    #pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.qfull[b], 1);
      mbar_init(&sm.qempty[b], kConsumerWarps);
      sm.uinfo[b].row = -1;  // "no unit": fails the consumers' range checks
    }
    sm.abort_flag = 0;
    sm.stop = 0;
    fence_barrier_init();
  }

  // ---- device plan, pass 1: total work of the decode-class rows ----------
  const int per = ceil_div(R, kDecodeThreads);
  const int r_lo = min(R, tid * per), r_hi = min(R, r_lo + per);
  long long work = 0;
  for (int r = r_lo; r < r_hi; ++r) {
    long long w;
    request_units(p, r, 0, &w);
    work += w;
    if (blockIdx.x == 0 && !request_ok(p, p.qsl[r], p.qsl[r + 1], p.seq_lens[r]))
      record_error(p.err, kErrBounds);
  }
  long long total_work;
  block_inclusive_scan<long long>(work, sm.red, &total_work);
  total_work *= Hkv;
  const int chunk = (int)max((long long)p.min_chunk,
                             (total_work + p.target_units - 1) / max(1, p.target_units));

  // ---- pass 2: units per request and their exclusive prefix sum ----------
  long long units = 0;
  for (int r = r_lo; r < r_hi; ++r) {
    long long w;
    units += request_units(p, r, chunk, &w);
  }
  long long total_units;
  const long long incl = block_inclusive_scan<long long>(units, sm.red, &total_units);
  {
    long long run = incl - units;
    for (int r = r_lo; r < r_hi; ++r) {
      prefix[r] = (int)run;
      long long w;
      run += request_units(p, r, chunk, &w);
    }
  }
  if (tid == 0) {
    if (total_units > p.max_units) {
      if (blockIdx.x == 0) record_error(p.err, kErrCapacity);
      total_units = 0;
    }
    prefix[R] = (int)total_units;
    sm.total_units = (int)total_units;
  }
  __syncthreads();
  const int T = sm.total_units;

  if (warp == kConsumerWarps) {
    // ======================= producer warp =================================
    const uint64_t pol = l2_policy_evict_first();
    int r = 0;
    uint32_t n = 0;  // CTA-wide block sequence number
    int j = 0;       // CTA-local unit index
    for (int u = blockIdx.x; u < T && !*abort_flag; u += gridDim.x, ++j) {
      while (r < R - 1 && prefix[r + 1] <= u) ++r;
      const int q0 = __ldg(p.qsl + r), qr = __ldg(p.qsl + r + 1) - q0;
      const int L = __ldg(p.seq_lens + r);
      const int nb = ceil_div(L, kBlockSize);
      const int S = ceil_div(nb, chunk);
      const int local = u - prefix[r];
      const int s = local % S;
      const int rest = local / S;
      const int k = rest % Hkv;
      const int i = rest / Hkv;
      const int limit = L - qr + i + 1;
      const int b0 = s * chunk;
      const int nblk = max(0, min(b0 + chunk, ceil_div(limit, kBlockSize)) - b0);
      const int ub = j & 1;
      if (j >= 2 && !mbar_wait(&sm.qempty[ub], ((j >> 1) - 1) & 1, p.err, abort_flag)) break;
      if (lane == 0) {
        UnitInfo ui;
        ui.row = q0 + i; ui.k = k; ui.b0 = b0; ui.nblk = nblk; ui.limit = limit;
        ui.S = S; ui.unit = u; ui.base = u - s;
        sm.uinfo[ub] = ui;
        mbar_arrive_expect_tx(&sm.qfull[ub], G * kHeadDim * 2);
        bulk_copy_g2s(sm.qbuf[ub],
                      p.q + ((long long)(q0 + i) * p.num_q_heads + (long long)k * G) * kHeadDim,
                      G * kHeadDim * 2, &sm.qfull[ub]);
      }
      const int32_t* bt = p.block_tables + (long long)r * p.max_blocks + b0;
      for (int bb = 0; bb < nblk && !*abort_flag; bb += 32) {
        const int cnt = min(32, nblk - bb);
        const int ent = lane < cnt ? __ldg(bt + bb + lane) : 0;
        for (int xb = 0; xb < cnt; ++xb, ++n) {
          int phys = __shfl_sync(0xffffffffu, ent, xb);
          const int st = n % kStages;
          if (n >= kStages && !mbar_wait(&sm.empty[st], ((n / kStages) - 1) & 1, p.err, abort_flag))
            break;
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
            bulk_copy_g2s(sm.ring[st] + kTileBytes, p.v_pool + tile, kTileBytes, &sm.full[st], pol);
          }
          __syncwarp();
        }
      }
    }
    return;
  }

  // ========================= consumer warps ================================
  using BM = BlockMath<G>;
  constexpr int F = BM::F;
  constexpr int kConsumerThreads = kConsumerWarps * 32;
  const int cw = warp;
  const int ct = tid;  // 0..127: the output dim this thread writes
  const int c = lane & 15;
  const int b0bit = lane & 1;
  uint32_t n_base = 0;
  int j = 0;
  for (int u = blockIdx.x; u < T; u += gridDim.x, ++j) {
    const int ub = j & 1;
    const bool have_q = mbar_wait(&sm.qfull[ub], (j >> 1) & 1, p.err, abort_flag);
    UnitInfo ui = sm.uinfo[ub];
    // Range checks make every later index safe even after an abort.
    const bool in_range = ui.row >= 0 && ui.row < p.num_q_tokens && ui.k >= 0 &&
                          ui.k < Hkv && ui.nblk >= 0 && ui.nblk <= p.max_blocks && ui.S >= 1 &&
                          ui.base >= 0 && ui.base + ui.S <= p.max_units && ui.unit >= ui.base &&
                          ui.unit < ui.base + ui.S;
    if (!(have_q && in_range)) ui.nblk = 0;
    float2 qf[G][4];
    #pragma unroll
    for (int hs = 0; hs < G; ++hs) {
      const int hl = BM::head_of_slot(hs, b0bit);
      const uint4 w = lds128(&sm.qbuf[ub][hl * kHeadDim + c * 8]);
      const float2 s2 = make_float2(p.scale_log2, p.scale_log2);
      qf[hs][0] = fmul2(bf16x2_to_float2(w.x), s2);
      qf[hs][1] = fmul2(bf16x2_to_float2(w.y), s2);
      qf[hs][2] = fmul2(bf16x2_to_float2(w.z), s2);
      qf[hs][3] = fmul2(bf16x2_to_float2(w.w), s2);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.qempty[ub]);

    float m[G], lsum[F];
    float2 acc[G][4];
    #pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = kNegBig;
      #pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = make_float2(0.f, 0.f);
    }
    #pragma unroll
    for (int jj = 0; jj < F; ++jj) lsum[jj] = 0.f;

    for (int bi = (int)((cw - n_base) & (kConsumerWarps - 1)); bi < ui.nblk; bi += kConsumerWarps) {
      const uint32_t n = n_base + bi;
      const int st = n % kStages;
      const bool arrived = mbar_wait(&sm.full[st], (n / kStages) & 1, p.err, abort_flag);
      const int first = (ui.b0 + bi) * kBlockSize;
      const int nvalid = (arrived && sm.stage_valid[st]) ? min(kBlockSize, ui.limit - first) : 0;
      BM::run(sm.ring[st], nvalid, lane, qf, m, lsum, acc, sm.pbuf[cw]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
    }
    n_base += ui.nblk;

    // ---- combine the four warps' states -----------------------------------
    float lall[G];
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
        for (int jj = 0; jj < G; ++jj) lall[jj] = l2[jj];
      }
    }
    #pragma unroll
    for (int h = 0; h < G; ++h)
      #pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[h][i].x += __shfl_xor_sync(0xffffffffu, acc[h][i].x, 16);
        acc[h][i].y += __shfl_xor_sync(0xffffffffu, acc[h][i].y, 16);
      }
    if (lane < 16) {
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        float4* dst = reinterpret_cast<float4*>(&sm.comb[cw][h][c * 8]);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
    }
    if (lane == 0) {
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        sm.comb_m[cw][h] = m[h];
        sm.comb_l[cw][h] = lall[h];
      }
      sm.wait_ok[cw] = have_q && in_range;
    }
    named_barrier(1, kConsumerThreads);

    // When every warp's wait succeeded, all four hold the same unit info (it
    // cannot change before all four have released the q buffer), so `ok` is
    // uniform across the consumer warps and so are the barriers below.
    bool ok = true;
    #pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) ok = ok && sm.wait_ok[w];
    const int d = ct;
    const long long out_row = ((long long)ui.row * p.num_q_heads + (long long)ui.k * G) * kHeadDim;
    float res[G];
    #pragma unroll
    for (int h = 0; h < G; ++h) {
      float M = sm.comb_m[0][h];
      #pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) M = fmaxf(M, sm.comb_m[w][h]);
      float num = 0.f, den = 0.f;
      #pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float e = fast_exp2(sm.comb_m[w][h] - M);
        num += e * sm.comb[w][h][d];
        den += e * sm.comb_l[w][h];
      }
      res[h] = den > 0.f ? num / den : 0.f;
      if (ok && ui.S > 1) {
        const long long slot = (long long)ui.unit * G + h;
        p.ws_o[slot * kHeadDim + d] = res[h];
        if (d == 0) {
          p.ws_ml[slot * 2] = M;
          p.ws_ml[slot * 2 + 1] = den;
        }
      }
    }
    if (ok && ui.S == 1) {
      #pragma unroll
      for (int h = 0; h < G; ++h) p.out[out_row + h * kHeadDim + d] = __float2bfloat16_rn(res[h]);
    }
    if (ok && ui.S > 1) {
      __threadfence();
      named_barrier(1, kConsumerThreads);
      if (ct == 0) {
        int* cnt = p.ws_cnt + (long long)ui.row * Hkv + ui.k;
        const int old = atomicAdd(cnt, 1);
        const int last = (old == ui.S - 1);
        if (last) *cnt = 0;  // every split has arrived: leave the counter at zero
        sm.is_last = last;
      }
      named_barrier(1, kConsumerThreads);
      if (sm.is_last) {
        // Log-sum-exp merge of the row's splits, in split order.
        __threadfence();
        #pragma unroll 1
        for (int h = 0; h < G; ++h) {
          float M = kNegBig;
          for (int s = 0; s < ui.S; ++s)
            M = fmaxf(M, __ldcg(p.ws_ml + ((long long)(ui.base + s) * G + h) * 2));
          float num = 0.f, den = 0.f;
          for (int s = 0; s < ui.S; ++s) {
            const long long slot = (long long)(ui.base + s) * G + h;
            const float w = fast_exp2(__ldcg(p.ws_ml + slot * 2) - M) * __ldcg(p.ws_ml + slot * 2 + 1);
            num += w * __ldcg(p.ws_o + slot * kHeadDim + d);
            den += w;
          }
          p.out[out_row + h * kHeadDim + d] = __float2bfloat16_rn(num / den);
        }
      }
    }
    // End of unit: agree on whether to stop (abort is set asynchronously, so
    // one thread samples it and the barrier publishes the sample).
    if (ct == 0) sm.stop = *abort_flag;
    named_barrier(1, kConsumerThreads);
    if (sm.stop) break;
  }
}

template <int G>
cudaError_t launch_decode_g(const DecodeParams& p, int sm_count, cudaStream_t stream) {
  const size_t smem = sizeof(DecodeSmem<G>) + (size_t)(p.num_reqs + 1) * sizeof(int);
  // The opt-in shared-memory limit is set once per device for the largest
  // plan (kMaxReqs requests).
  static unsigned long long configured = 0;  // bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(DecodeSmem<G>) + (kMaxReqs + 1) * sizeof(int)));
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<G>, kDecodeThreads, smem);
  if (e != cudaSuccess) return e;
  per_sm = max(1, per_sm);
  const int grid = max(1, min(p.max_units, sm_count * per_sm));
  decode_kernel<G><<<grid, kDecodeThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_target_units(int sm_count) { return sm_count * 4; }

WorkspaceLayout decode_workspace_layout(int num_q_tokens, int num_kv_heads, int group,
                                        int target_units) {
  WorkspaceLayout w;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  w.max_units = target_units + num_q_tokens * num_kv_heads;
  w.cnt_off = 0;
  w.ml_off = up((size_t)num_q_tokens * num_kv_heads * sizeof(int));
  w.o_off = w.ml_off + up((size_t)w.max_units * group * 2 * sizeof(float));
  w.total = w.o_off + up((size_t)w.max_units * group * kHeadDim * sizeof(float));
  return w;
}

cudaError_t launch_decode(const DecodeParams& p, int group, int sm_count, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_g<1>(p, sm_count, stream);
    case 2: return launch_decode_g<2>(p, sm_count, stream);
    case 3: return launch_decode_g<3>(p, sm_count, stream);
    case 4: return launch_decode_g<4>(p, sm_count, stream);
    case 5: return launch_decode_g<5>(p, sm_count, stream);
    case 6: return launch_decode_g<6>(p, sm_count, stream);
    case 7: return launch_decode_g<7>(p, sm_count, stream);
    case 8: return launch_decode_g<8>(p, sm_count, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
