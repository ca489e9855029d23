// pkv_prefill.cu -- ragged chunked-prefill attention on tcgen05 tensor cores.
//
// A prefill chunk of q_r query tokens attends causally to the keys earlier
// chunks wrote plus its own (The Serving Playbook, "Chunked prefill"); with
// many query rows per request the step is a real dense contraction, so QK^T
// and PV run on the 5th-generation tensor cores with fp32 accumulators in
// TMEM, FlashAttention-style: Q, K and V tiles are staged in shared memory,
// the score matrix never leaves the chip, and an online softmax carries the
// running maximum and normaliser across key tiles (LLM 7 - Efficient LLM
// Serving, sec. 2).
//
// Tiling.  A work item is (request, KV head, q-tile).  Its 128 MMA rows are
// (query token, head of the group) pairs -- T_q = floor(128 / g) tokens times
// the g query heads that share the KV head -- so every K/V tile loaded for
// the item serves all g heads.  Key tiles are 128 keys = 8 pool blocks; each
// 16-row block tile is fetched through the block table with a 2-D TMA copy
// of the pool viewed as [blocks * Hkv * 16 rows, 128] (128-byte swizzle);
// blocks past the request's end are fetched at an out-of-range row, which TMA
// fills with zeros.  Q comes in with one 3-D TMA copy per half (d, head,
// token).
//
// Roles (608 threads): sixteen softmax warps -- warps 0-15, four threads
// per TMEM lane / MMA row, each taking a quarter of the row's keys and of
// its output dims -- run the softmax and the epilogue; warp 16 takes items
// from a work queue in the workspace and issues the Q and K copies, warp 18
// the V copies of the items warp 16 hands it; one thread of warp 17 issues
// tcgen05.mma and commits.  Four threads per row (rather than two) halve each
// thread's serial chain of exponentials per tile and double the warps that
// hide its latencies: the softmax, not the tensor core, sets the pace.
// Per key tile: S = Q K^T (8 MMAs of K=16) into TMEM, the softmax reads S and
// writes P (bf16, two keys per column) over it, then O += P V (8 MMAs, A read
// from TMEM) accumulates in TMEM.  K and V have rings of their own: a K stage
// is free once its QK^T is done, a V stage once its PV is, so K runs ahead of
// the tensor core by the whole ring.  O is rescaled in TMEM only when a row's
// maximum grows by more than 2^8 (the result is exact either way: O and the
// normaliser always share the same reference maximum).
#include <climits>

#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kParts = 4;                // softmax threads per MMA row
constexpr int kPartKeys = 128 / kParts;  // keys (and output dims) per softmax thread
constexpr int kSoftWarps = 4 * kParts;   // warps 0 .. 15
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kWarpQK = kSoftWarps;      // Q + K producer (takes the items)
constexpr int kWarpMma = kSoftWarps + 1; // MMA issuer
constexpr int kWarpV = kSoftWarps + 2;   // V producer
constexpr int kPfThreads = 32 * (kSoftWarps + 3);
constexpr int kBarSoftmax = 1;           // the softmax warps' named barrier
constexpr int kBarQuad = 2;              // + quad: the four warps holding the same 32 rows
constexpr int kTileRows = 128;               // MMA M
constexpr int kKeyTile = 128;                // MMA N for S, K for PV
constexpr int kHalfBytes = kTileRows * 128;  // one 64-column half of a 128-row tile
constexpr uint32_t kTmemCols = 512;          // S0: cols 0..127, S1: 128..255, O: 256..383
constexpr float kRescaleLog2 = 8.0f;
constexpr float kNegBig = -1.0e30f;
// Debug-only per-tile timeline of CTA 0 (build with -DPKV_PF_TRACE=1):
// %globaltimer at load issue, keys seen by the MMA warp, scores seen by the
// softmax, probabilities ready (PV issue), stage released to the producer;
// then, for the softmax thread of row 0, key part 0: scores in registers,
// vote done, exponentials done, P stored in TMEM, arrival.
#ifndef PKV_PF_TRACE
#define PKV_PF_TRACE 0
#endif
#if PKV_PF_TRACE
constexpr int kPfTrTiles = 64;
__device__ unsigned long long g_pf_trace[10][kPfTrTiles];
#define PF_TR(ev, tile) do { if (blockIdx.x == 0 && (tile) < kPfTrTiles) g_pf_trace[ev][tile] = global_timer_ns(); } while (0)
#else
#define PF_TR(ev, tile) do { } while (0)
#endif
constexpr int kPastEnd = INT_MIN;            // block-table slot past the request (not read)

struct Item {
  int r, k;   // block-table row, KV head
  int row0;   // first query row of the tile
  int nt;     // valid tokens in the tile
  int pos0;   // position of its first token
  int L;      // request length (keys)
  int nj;     // key tiles
  int causal; // 0: prefix pass (every row sees all L keys)
  int kt0;    // first key tile (a prefix-pass chunk of the keys)
  int kc;     // prefix-pass chunk index (selects the partial-state slot)
  int end;    // no more items
};

// K and V tile stages (32 KiB each).  A V tile is needed only after its
// tile's softmax, so its ring can be one stage shorter than K's; the room
// holds the softmax threads' row exchange.
constexpr int kPfStagesK = 3;
constexpr int kPfStagesV = 2;

struct __align__(1024) PfSmem {
  uint8_t q[2][kHalfBytes];              // Q: d 0..63 | d 64..127
  uint8_t k[kPfStagesK][2][kHalfBytes];  // [stage][d half]
  uint8_t v[kPfStagesV][2][kHalfBytes];  // [stage][d half]
  uint64_t q_full, q_empty;
  uint64_t k_full[kPfStagesK], v_full[kPfStagesV], k_empty[kPfStagesK], v_empty[kPfStagesV];
  uint64_t s_full[2], p_full[2], p_free[2];
  uint64_t o_full, o_empty;
  Item items[2];
  float xrow[kParts][kTileRows]; // [key part][row]: partial row maxima, then normalisers
  Item vitems[4];                // items handed from the K producer to the V producer
  uint64_t vitem_full[4], vitem_empty[4];
  uint32_t tmem_base;
  WaitCtl wait;                   // abort flag and wait limit of the bounded waits
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// A unit of prefill work: a request's query chunk (causal over its keys), or
// in the prefix pass a sharing group's query tokens against its shared
// blocks (every key visible).
struct PfReq {
  int q0, qr, L, ntiles;  // ntiles: items per KV head (q-tiles x key chunks)
  int tab;     // block-table row
  int nchunk;  // key chunks (prefix pass; 1 otherwise)
  bool ok;
};

__device__ __forceinline__ int num_units(const PrefillParams& p) {
  return p.prefix_mode ? p.num_groups : p.num_reqs;
}

__device__ __forceinline__ PfReq load_pf_request(const PrefillParams& p, int u, int tq) {
  PfReq a;
  if (p.prefix_mode) {
    const int first = __ldg(p.grp_first + u), n = __ldg(p.grp_count + u);
    const int nb = __ldg(p.grp_blocks + u);
    const bool idx_ok = first >= 0 && n >= 1 && (long long)first + n <= p.num_reqs;
    a.tab = idx_ok ? first : 0;
    a.q0 = idx_ok ? __ldg(p.qsl + first) : 0;
    const int q1 = idx_ok ? __ldg(p.qsl + first + n) : 0;
    a.qr = q1 - a.q0;
    a.L = nb * kBlockSize;
    a.ok = idx_ok && a.q0 >= 0 && a.qr >= 1 && q1 <= p.num_q_tokens && nb >= 1 &&
           nb <= p.max_blocks;
  } else {
    a.tab = u;
    a.q0 = __ldg(p.qsl + u);
    const int q1 = __ldg(p.qsl + u + 1);
    a.L = __ldg(p.seq_lens + u);
    a.qr = q1 - a.q0;
    a.ok = a.q0 >= 0 && a.qr >= p.prefill_min_q && q1 <= p.num_q_tokens && a.qr <= a.L &&
           a.L <= p.max_blocks * kBlockSize;
  }
  a.nchunk = p.prefix_mode ? prefix_chunks(a.L) : 1;
  a.ntiles = a.ok ? ceil_div(a.qr, tq) * a.nchunk : 0;
  return a;
}

// Rarely run parts of the softmax warps, out of line: one copy each keeps
// the kernel's instruction footprint small.
// O (this thread's 32 output columns at TMEM address tO) times alpha.
static __device__ __noinline__ void rescale_o32(uint32_t tO, float alpha) {
  float o[32];
  tmem_ld32(tO, o);
  tc_wait_ld();
  #pragma unroll
  for (int i = 0; i < 32; ++i) o[i] *= alpha;
  tmem_st32(tO, o);
  tc_wait_st();
}

// Zeroes rows tail0 .. tail0 + nrows - 1 of a staged V tile (two 64-column
// halves `half_bytes` apart, 128-byte swizzled); warp-collective.
static __device__ __noinline__ void zero_v_rows(uint8_t* v, int half_bytes, int tail0, int nrows,
                                                int lane) {
  for (int i = lane; i < nrows * 16; i += 32) {
    const int rr = tail0 + i / 16, hf = (i / 8) & 1, chunk = i & 7;
    *reinterpret_cast<uint4*>(v + hf * half_bytes + (rr >> 3) * 1024 + (rr & 7) * 128 +
                              chunk * 16) = make_uint4(0, 0, 0, 0);
  }
}

template <int G>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  constexpr int TQ = kTileRows / G;   // query tokens per item
  constexpr int ROWS = TQ * G;        // MMA rows in use
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled tiles need 1024-byte aligned shared addresses.
  const uint32_t raw = smem_u32(smem_raw);
  PfSmem& sm = *reinterpret_cast<PfSmem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  WaitCtl* abort_flag = &sm.wait;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.num_kv_heads;

  // Ordering.  The decode kernel launched just before this one in the same
  // call lets it start early; everything read here (lengths, tables, q, the
  // pools) was complete before the decode kernel signalled, and the decode
  // kernel writes only decode rows of `out`, which this kernel never touches.
  // So the work below needs no wait; the wait at the end makes this grid
  // finish after the decode grid, so that successors of the call see both.
  //
  // Before any set-up: does this CTA have an item at all?  Pure-decode steps
  // (no request with q_r >= prefill_min_q) leave every CTA idle.
  if (warp == 0) {
    long long total = 0;
    for (int b = 0; b < num_units(p); b += 32) {
      const int rr = b + lane;
      long long cnt = 0;
      if (rr < num_units(p)) cnt = (long long)load_pf_request(p, rr, TQ).ntiles * Hkv;
      #pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      total += cnt;
    }
    if (lane == 0) {
      sm.wait.abort = (long long)blockIdx.x >= total;  // reused as "idle"
      sm.items[0].r = (int)min(total, (long long)gridDim.x);  // CTAs that take items
    }
  }
  __syncthreads();
  if (sm.wait.abort) {
    allow_dependent_launch();
    grid_dependency_wait();
    return;
  }
  const int n_active = sm.items[0].r;
  __syncthreads();

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < kPfStagesK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kPfStagesV; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);   // tcgen05.commit after S = QK^T into buffer b
      mbar_init(&sm.p_full[b], kSoftWarps);  // P written over S buffer b (and O rescaled)
      mbar_init(&sm.p_free[b], 1);   // tcgen05.commit after the PV that read P in buffer b
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_empty, kSoftWarps);
    for (int b = 0; b < 4; ++b) {
      mbar_init(&sm.vitem_full[b], 1);
      mbar_init(&sm.vitem_empty[b], 1);
    }
    sm.wait.abort = 0;
    sm.wait.limit_ns = p.wait_limit_ns;
    fence_barrier_init();
  }
  if (warp == kWarpQK && lane == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  // Q rows no item writes stay zero (their S and O rows are never read).
  if constexpr (ROWS < kTileRows) {
    constexpr int kPad = (kTileRows - ROWS) * 8;  // 16-byte chunks per half
    for (int i = tid; i < 2 * kPad; i += kPfThreads) {
      const int half = i / kPad;
      const int rest = i % kPad;
      const int row = ROWS + rest / 8, chunk = rest % 8;
      *reinterpret_cast<uint4*>(sm.q[half] + (row / 8) * 1024 + (row % 8) * 128 + chunk * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  allow_dependent_launch();

  if (warp == kWarpQK || warp == kWarpV) {
    // ==================== TMA producers (K + Q | V) =======================
    // Warp 16 takes items from the work queue, streams their K tiles and Q,
    // and hands each item to warp 18, which streams the V tiles.
    const bool vside = warp == kWarpV;
    uint64_t* const full = vside ? sm.v_full : sm.k_full;
    uint64_t* const empty = vside ? sm.v_empty : sm.k_empty;
    const CUtensorMap* const map = vside ? &vmap : &kmap;
    int n_item = 0, tile_ctr = 0;
    const int oob_row = p.num_blocks * Hkv * kBlockSize;
    // The item's tiles (and, on the K side, its Q).  False if a wait gave up.
    auto stream_item = [&](const Item& it) {
      const int nbl = ceil_div(it.L, kBlockSize);
      const int32_t* bt = p.block_tables + (long long)it.r * p.max_blocks;
      // Block-table entries 32 blocks (four key tiles) per load, the next
      // group fetched while the current one is issued, checked at use.
      auto raw_entries = [&](int x0) {
        const int x = it.kt0 * 8 + x0 + lane;
        return x < nbl ? __ldg(bt + x) : kPastEnd;
      };
      int ent_cur = raw_entries(0);
      int ent_nxt = it.nj > 4 ? raw_entries(32) : kPastEnd;
      for (int j = 0; j < it.nj; ++j, ++tile_ctr) {
        if (j > 0 && (j & 3) == 0) {
          ent_cur = ent_nxt;
          if (j + 4 < it.nj) ent_nxt = raw_entries((j + 4) * 8);
        }
        const int stages = vside ? kPfStagesV : kPfStagesK;
        const int st = tile_ctr % stages;
        if (tile_ctr >= stages &&
            !mbar_wait(&empty[st], ((tile_ctr / stages) - 1) & 1, p.err, abort_flag))
          return false;
        if (lane == 0 && vside && tile_ctr >= stages) PF_TR(4, tile_ctr - stages);
        if (lane == 0 && !vside) PF_TR(0, tile_ctr);
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 2u * kHalfBytes);
        __syncwarp();
        // Lanes 0..15 each copy one (block, d half); blocks past the
        // request are read at an out-of-range row (zero fill).
        const int bsel = lane & 7, hsel = (lane >> 3) & 1;
        const int phys = __shfl_sync(0xffffffffu, ent_cur, (j & 3) * 8 + bsel);
        if (lane < 16) {
          int rowc = oob_row;
          if ((unsigned)phys < (unsigned)p.num_blocks) rowc = (phys * Hkv + it.k) * kBlockSize;
          else if (phys != kPastEnd && hsel == 0 && !vside) record_error(p.err, kErrBounds);
          uint8_t* dst = (vside ? sm.v[st][hsel] : sm.k[st][hsel]) + bsel * 2048;
          tma_load_2d(dst, map, hsel * 64, rowc, &full[st]);
        }
        __syncwarp();
        if (j == 0 && !vside) {
          // Q of this item, once the previous item's MMAs are done with Q
          // (its first K tile is already on its way).
          if (n_item >= 1 && !mbar_wait(&sm.q_empty, (n_item - 1) & 1, p.err, abort_flag))
            return false;
          if (lane == 0) {
            sm.items[n_item & 1] = it;
            mbar_arrive_expect_tx(&sm.q_full, 2u * 64u * ROWS * 2u);
            tma_load_3d(sm.q[0], &qmap, 0, it.k * G, it.row0, &sm.q_full);
            tma_load_3d(sm.q[1], &qmap, 64, it.k * G, it.row0, &sm.q_full);
          }
          __syncwarp();
        }
      }
      return true;
    };
    if (vside) {
      for (;; ++n_item) {
        const int mb = n_item & 3;
        if (!mbar_wait(&sm.vitem_full[mb], (n_item >> 2) & 1, p.err, abort_flag)) break;
        const Item it = sm.vitems[mb];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.vitem_empty[mb]);
        if (it.end || !stream_item(it)) break;
      }
    } else {
      // Items are numbered batch of 32 requests by batch, request by request
      // within a batch (longest first; heavier q-tiles first within a
      // request), and taken from the queue in that order, so each CTA's
      // sequence increases and one forward scan over the batches serves it.
      auto next_item = [&]() {
        unsigned long long v = 0;
        if (lane == 0) v = atomicAdd(p.sched, 1ull);
        return (long long)__shfl_sync(0xffffffffu, v, 0);
      };
      auto hand_over = [&](const Item& it) {  // to the V producer
        const int mb = n_item & 3;
        if (n_item >= 4 &&
            !mbar_wait(&sm.vitem_empty[mb], ((n_item >> 2) - 1) & 1, p.err, abort_flag))
          return false;
        if (lane == 0) {
          sm.vitems[mb] = it;
          mbar_arrive(&sm.vitem_full[mb]);
        }
        __syncwarp();
        return true;
      };
      long long item = next_item();  // global item index handled next
      long long base = 0;            // items before the current request batch
      const int nunits = num_units(p);
      bool ok = true;
      for (int b = 0; b < nunits && ok && !abort_flag->abort; b += 32) {
        const int rr = b + lane;
        PfReq rq = {0, 0, 0, 0, 0, 1, false};
        if (rr < nunits) rq = load_pf_request(p, rr, TQ);
        const long long cnt = (long long)rq.ntiles * Hkv;
        long long total = cnt;
        #pragma unroll
        for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
        if (item >= base + total) {  // no item of this batch left for this CTA
          base += total;
          continue;
        }
        // Within a batch of 32 requests the longest go first (then by index):
        // a request's items cost about L / 128 key tiles each, and taking
        // the longest first leaves short items for the queue's end, where
        // the CTAs run out of work at different times.
        const int key = cnt > 0 ? rq.L : -1;
        long long excl = 0;
        #pragma unroll 4
        for (int s = 0; s < 32; ++s) {
          const int ks = __shfl_sync(0xffffffffu, key, s);
          const long long cs = __shfl_sync(0xffffffffu, cnt, s);
          if (ks > key || (ks == key && s < lane)) excl += cs;
        }
        const long long incl = excl + cnt;
        while (item < base + total && ok && !abort_flag->abort) {
          const long long rel = item - base;
          const unsigned own = __ballot_sync(0xffffffffu, cnt > 0 && excl <= rel && rel < incl);
          const int src = __ffs(own) - 1;
          const long long local = rel - __shfl_sync(0xffffffffu, excl, src);
          const int r = __shfl_sync(0xffffffffu, rq.tab, src);
          const int q0 = __shfl_sync(0xffffffffu, rq.q0, src);
          const int qr = __shfl_sync(0xffffffffu, rq.qr, src);
          const int L = __shfl_sync(0xffffffffu, rq.L, src);
          const int ntiles = __shfl_sync(0xffffffffu, rq.ntiles, src);
          const int nchunk = __shfl_sync(0xffffffffu, rq.nchunk, src);
          // heavier (later) q-tiles first
          const int qk = ntiles - 1 - (int)(local / Hkv);
          const int qt = qk / nchunk, kc = qk % nchunk;
          Item it;
          it.r = r;
          it.k = (int)(local % Hkv);
          it.row0 = q0 + qt * TQ;
          it.nt = min(TQ, qr - qt * TQ);
          it.pos0 = L - qr + qt * TQ;
          it.L = L;
          it.causal = !p.prefix_mode;
          it.kc = kc;
          it.kt0 = it.causal ? 0 : kc * prefix_chunk_tiles(L);
          it.nj = it.causal ? (it.pos0 + it.nt - 1) / kKeyTile + 1
                            : min(prefix_chunk_tiles(L), ceil_div(L, kKeyTile) - it.kt0);
          it.end = 0;
          ok = hand_over(it) && stream_item(it);
          ++n_item;
          item = next_item();
        }
        base += total;
      }
      // end markers: for the V producer, and for the MMA and softmax warps
      // (the Q side owns the item slots)
      Item fin = {};
      fin.end = 1;
      if (ok) hand_over(fin);
      if (n_item == 0 || mbar_wait(&sm.q_empty, (n_item - 1) & 1, p.err, abort_flag)) {
        if (lane == 0) {
          sm.items[n_item & 1].end = 1;
          mbar_arrive(&sm.q_full);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ========================= MMA issuer =================================
    // Tile t: S(t) = Q K(t)^T into S buffer t&1, then O += P(t-1) V(t-1).  S
    // of the next tile therefore runs on the tensor core while the softmax
    // warps work on the current one.
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTileRows, kKeyTile, 0, 0);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTileRows, kHeadDim, 0, 1);
      const uint32_t tO = tmem + 2 * kKeyTile;
      int t = 0;  // tile counter, shared sequence with the producer and softmax
      bool ok = true;
      auto pv = [&](int tt, bool first, int n_item) {
        const int b = tt & 1, st = tt % kPfStagesV;
        ok = ok && mbar_wait(&sm.p_full[b], (tt >> 1) & 1, p.err, abort_flag);
        ok = ok && mbar_wait(&sm.v_full[st], (tt / kPfStagesV) & 1, p.err, abort_flag);
        if (first && n_item > 0)
          ok = ok && mbar_wait(&sm.o_empty, (n_item - 1) & 1, p.err, abort_flag);
        PF_TR(3, tt);
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // P (bf16) lies in the first 64 columns of S buffer b, two keys
          // per column: keys 16kk .. 16kk+15 in columns 8kk .. 8kk+7.
          const uint32_t ta = tmem + b * kKeyTile + kk * 8;
          // V is MN-major (d contiguous): atoms of 64 d x 8 keys; the two d
          // halves are kHalfBytes apart, 8-key groups 1024 bytes apart.
          const uint64_t db = smem_desc_sw128(smem_u32(sm.v[st][0]) + kk * 2048, kHalfBytes, 1024);
          tc_mma_f16_ts(tO, ta, db, kIdescO, !first || kk > 0);
        }
        tc_commit(&sm.v_empty[st]);
        tc_commit(&sm.p_free[b]);
      };
      for (int n_item = 0; ok; ++n_item) {
        if (!mbar_wait(&sm.q_full, n_item & 1, p.err, abort_flag)) break;
        const Item it = sm.items[n_item & 1];
        if (it.end) break;
        tc_fence_after();
        for (int j = 0; j < it.nj && ok; ++j, ++t) {
          const int b = t & 1, st = t % kPfStagesK;
          ok = ok && mbar_wait(&sm.k_full[st], (t / kPfStagesK) & 1, p.err, abort_flag);
          PF_TR(1, t);
          // S buffer b holds P(t - 2) until the PV of tile t - 2 has read it.
          if (t >= 2) ok = ok && mbar_wait(&sm.p_free[b], ((t >> 1) - 1) & 1, p.err, abort_flag);
          tc_fence_after();
          const uint32_t tS = tmem + b * kKeyTile;
          #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t da = smem_desc_sw128(smem_u32(sm.q[kk >> 2]) + (kk & 3) * 32, 16, 1024);
            const uint64_t db = smem_desc_sw128(smem_u32(sm.k[st][kk >> 2]) + (kk & 3) * 32, 16, 1024);
            tc_mma_f16_ss(tS, da, db, kIdescS, kk > 0);
          }
          tc_commit(&sm.k_empty[st]);
          tc_commit(&sm.s_full[b]);
          if (j >= 1) pv(t - 1, j == 1, n_item);
        }
        if (ok) pv(t - 1, it.nj == 1, n_item);  // the item's last tile
        tc_commit(&sm.o_full);
        tc_commit(&sm.q_empty);
      }
    }
    __syncwarp();
  } else if (warp < kSoftWarps) {
    // =================== softmax + epilogue (warps 0-15) =====================
    // Four threads share each MMA row: warps 4c .. 4c+3 take keys 32c .. 32c+31
    // of a tile and output dims 32c .. 32c+31.  Warp w reaches TMEM lanes
    // 32 (w % 4) .. +31, so the four warps with equal w % 4 hold the same 32
    // rows.  The four parts agree on the row maximum through shared memory
    // once per tile.
    const int quad = warp & 3;
    const int part = warp >> 2;
    const int row = quad * 32 + lane;  // MMA row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tO = tmem + lane_off + 2 * kKeyTile + part * kPartKeys;
    const int t_local = row / G, h = row % G;
    int tile_ctr = 0;
    for (int n_item = 0;; ++n_item) {
      const bool have = mbar_wait(&sm.q_full, n_item & 1, p.err, abort_flag);
      const Item it = sm.items[n_item & 1];
      // Agree before any barrier: a wait that gave up (abort) stops everyone.
      if (barrier_or(kBarSoftmax, kSoftThreads, !have || it.end)) break;
      const bool valid = row < ROWS && t_local < it.nt;
      // The last key this row sees (all keys in the prefix pass).
      const int prow = !valid ? -1 : it.causal ? it.pos0 + t_local : it.L - 1;
      float m = kNegBig, l = 0.f;
      bool ok = true;
      for (int j = 0; j < it.nj; ++j, ++tile_ctr) {
        const int sb = tile_ctr & 1;  // S / P buffer of this tile
        const uint32_t tS = tmem + lane_off + sb * kKeyTile;
        ok = ok && mbar_wait(&sm.s_full[sb], (tile_ctr >> 1) & 1, p.err, abort_flag);
        if (row == 0 && part == 0) PF_TR(2, tile_ctr);
        tc_fence_after();
        // This part's 32 scores, read from TMEM once, and their maximum over
        // the visible keys.
        const int kbase = (it.kt0 + j) * kKeyTile + part * kPartKeys;
        const bool full_part = kbase + kPartKeys - 1 <= prow;  // no key of this part masked
        float v[kPartKeys];
        tmem_ld32(tS + part * kPartKeys, v);
        tc_wait_ld();
        if (row == 0 && part == 0) PF_TR(5, tile_ctr);
        if (!full_part) {
          #pragma unroll
          for (int i = 0; i < kPartKeys; ++i)
            if (kbase + i > prow) v[i] = -INFINITY;
        }
        float mxp[4];
        #pragma unroll
        for (int i = 0; i < 4; ++i) mxp[i] = -INFINITY;
        #pragma unroll
        for (int i = 0; i < kPartKeys / 2; ++i) mxp[i & 3] = fmax3(mxp[i & 3], v[2 * i], v[2 * i + 1]);
        const float mxh = fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])) * p.scale_log2;
        // Past an item's first tile the row maximum is needed only when some
        // part's scores exceed the reference by more than 2^8: a vote of the
        // four warps that hold these rows decides, and only then do the parts
        // exchange their maxima.  The vote (a barrier of those warps) also
        // orders their S reads before any P write (P of part c lands in TMEM
        // columns that held the scores of keys 16c .. 16c + 15, of the same
        // rows).  Each group of rows keeps its own pace: the PV waits for all.
        tc_fence_before();
        const bool exchange = barrier_or(kBarQuad + quad, 128, j == 0 || mxh > m + kRescaleLog2);
        tc_fence_after();
        if (row == 0 && part == 0) PF_TR(6, tile_ctr);
        float mx = mxh;
        if (exchange) {
          sm.xrow[part][row] = mxh;
          named_barrier(kBarQuad + quad, 128);
          mx = fmaxf(fmaxf(sm.xrow[0][row], sm.xrow[1][row]),
                     fmaxf(sm.xrow[2][row], sm.xrow[3][row]));
          named_barrier(kBarQuad + quad, 128);  // sm.xrow is free again
        }
        float m_use = m;
        const bool grow = exchange && (j == 0 || mx > m + kRescaleLog2);
        if (j == 0) {
          m_use = fmaxf(m, mx);
        } else if (__any_sync(0xffffffffu, grow)) {
          // O (and l) move to the new reference maximum; rows that do not
          // grow scale by 1.  O must first hold the previous tile's PV.
          ok = ok && mbar_wait(&sm.p_free[(tile_ctr - 1) & 1], ((tile_ctr - 1) >> 1) & 1, p.err,
                               abort_flag);
          tc_fence_after();
          const float m_new = grow ? fmaxf(m, mx) : m;
          const float alpha = fast_exp2(m - m_new);
          rescale_o32(tO, alpha);
          l *= alpha;
          m_use = m_new;
        }
        m = m_use;
        // P = exp2(s * scale_log2 - m) in bf16 (masked keys are -inf: p = 0),
        // written over the row's S in TMEM two keys per column -- keys
        // 32 part .. +31 in columns 16 part .. +15 -- where the PV MMA reads
        // it; the normaliser sums the rounded values the MMA will use.  Pairs
        // of keys go through packed fp32 arithmetic.
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m, -m);
        float sum_lo[2] = {0.f, 0.f}, sum_hi[2] = {0.f, 0.f};
        uint32_t w[kPartKeys / 2];
        #pragma unroll
        for (int e = 0; e < kPartKeys / 2; ++e) {
          const float2 x = ffma2(make_float2(v[2 * e], v[2 * e + 1]), sc2, nm2);
          w[e] = pack_bf16x2(fast_exp2(x.x), fast_exp2(x.y));
          add_bf16x2(sum_lo[e & 1], sum_hi[e & 1], w[e]);
        }
        if (row == 0 && part == 0) PF_TR(7, tile_ctr);
        tmem_st16(tS + part * (kPartKeys / 2), w);
        tc_wait_st();
        if (row == 0 && part == 0) PF_TR(8, tile_ctr);
        l += (sum_lo[0] + sum_hi[0]) + (sum_lo[1] + sum_hi[1]);
        // Keys past the request's end inside its last block may hold anything
        // (even NaN); zero those V rows so that 0 * V stays 0 in the MMA.
        const int st = tile_ctr % kPfStagesV;
        const int tbase = (it.kt0 + j) * kKeyTile;
        const int tail0 = it.L - tbase;                      // first key >= L in this tile
        const int tail1 = min(kKeyTile, ceil_div(it.L, kBlockSize) * kBlockSize - tbase);
        if (warp == 0 && tail0 < tail1 && tail0 >= 0) {
          ok = ok && mbar_wait(&sm.v_full[st], (tile_ctr / kPfStagesV) & 1, p.err, abort_flag);
          zero_v_rows(sm.v[st][0], (int)(sm.v[st][1] - sm.v[st][0]), tail0, tail1 - tail0, lane);
          fence_proxy_async_smem();  // the zeros, read by the tensor core
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[sb]);
        if (row == 0 && part == 0) PF_TR(9, tile_ctr);
      }
      // ---- epilogue: O / l -> bf16 -> out (this part's 32 dims) ----------
      sm.xrow[part][row] = l;
      named_barrier(kBarQuad + quad, 128);
      const float lrow = (sm.xrow[0][row] + sm.xrow[1][row]) + (sm.xrow[2][row] + sm.xrow[3][row]);
      named_barrier(kBarQuad + quad, 128);  // sm.xrow is free again
      ok = ok && mbar_wait(&sm.o_full, n_item & 1, p.err, abort_flag);
      tc_fence_after();
      const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
      const long long orow = (long long)(it.row0 + t_local) * p.num_q_heads + (long long)it.k * G + h;
      __nv_bfloat16* dst = p.out + orow * kHeadDim + part * kPartKeys;
      // Prefix pass: the partial state of this key chunk.
      const long long prow_slot = (long long)it.kc * p.num_q_tokens * p.num_q_heads + orow;
      float* pdst = p.pre_o + prow_slot * kHeadDim + part * kPartKeys;
      if (p.prefix_mode && valid && ok && part == 0)
        *reinterpret_cast<float2*>(p.pre_ml + prow_slot * 2) = make_float2(m, lrow);
      {
        float o[32];
        tmem_ld32(tO, o);
        tc_wait_ld();
        if (valid && ok && p.prefix_mode) {
          #pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(pdst + i) =
                make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
        } else if (valid && ok) {
          #pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 q4;
            q4.x = pack_bf16x2(o[i] * inv, o[i + 1] * inv);
            q4.y = pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv);
            q4.z = pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv);
            q4.w = pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv);
            *reinterpret_cast<uint4*>(dst + i) = q4;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.o_empty);
    }
  }
  // Every warp reaches this point (aborts only shorten the loops), so the
  // allocating warp can always free TMEM.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
  grid_dependency_wait();
  // The last CTA to finish empties the work queue for the next launch (each
  // CTA stops taking items before it gets here).
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1ull) == (unsigned long long)(n_active - 1)) {
      p.sched[0] = 0;
      p.sched[1] = 0;
      __threadfence();
    }
  }
}

static_assert(sizeof(PfSmem) + 1024 <= 227 * 1024, "prefill shared memory");

template <int G>
cudaError_t launch_prefill_g(const PrefillLaunch& L, cudaStream_t stream) {
  const size_t smem = sizeof(PfSmem) + 1024;  // + alignment slack
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(prefill_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_kernel<G>, L.qmap, L.kmap, L.vmap, L.p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int prefill_tokens_per_tile(int group) { return kTileRows / group; }

#if PKV_PF_TRACE
cudaError_t prefill_trace(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_pf_trace, bytes < sizeof(g_pf_trace) ? bytes : sizeof(g_pf_trace));
}
#endif

cudaError_t launch_prefill(const PrefillLaunch& L, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefill_g<1>(L, stream);
    case 2: return launch_prefill_g<2>(L, stream);
    case 3: return launch_prefill_g<3>(L, stream);
    case 4: return launch_prefill_g<4>(L, stream);
    case 5: return launch_prefill_g<5>(L, stream);
    case 6: return launch_prefill_g<6>(L, stream);
    case 7: return launch_prefill_g<7>(L, stream);
    case 8: return launch_prefill_g<8>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
