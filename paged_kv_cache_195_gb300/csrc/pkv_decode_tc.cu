// pkv_decode_tc.cu -- paged decode attention on tcgen05 tensor cores, for
// GQA groups of g >= 4 query heads per KV head.
//
// What it computes is the decode kernel's (pkv_decode_kernel.cuh): for every
// query row served by the decode path and every KV head, the softmax-weighted
// sum of V over the row's visible keys, gathered through the block table (The
// Serving Playbook, "The block table lives in the hottest kernel in the
// system"), with an fp32 online softmax (LLM 7 - Efficient LLM Serving,
// sec. 2 "Online Softmax Makes Tiling Possible") and a log-sum-exp merge of
// the pieces a row is split into (The Serving Playbook, "Kernel fusion,
// briefly").  The work plan -- equal contiguous ranges of the step's block
// sequence, one per CTA -- is the same (pkv_plan.cuh), and so is the
// workspace format of partial pieces.
//
// Why tensor cores.  With g heads sharing a KV head, each K or V element
// feeds g multiply-adds per query row: 2g FMAs per 2-byte element.  GB300's
// FP32 pipe peaks near 128 FMA/clk/SM, so at g = 6 the FMA work of a block
// is half its HBM time at the copy peak, and an e4m3 cache would need all of
// it.  The group's QK^T and PV are small dense contractions; run them on the
// tensor core instead and the SIMT work left per key is one exp2 per head.
//
// Shape.  A tile is 128 consecutive keys of a piece = 8 pool blocks, each
// (block, KV head) 16-row slab fetched through the block table by a 2-D TMA
// copy (128-byte swizzle; blocks past the piece are fetched at an
// out-of-range row, which TMA fills with zeros).  With the keys as the MMA's
// M dimension and the group's heads as N (padded to 16):
//     S^T[128 keys x 16] = K[128 x 128 d] . Q^T                 (K-major A, B)
//     O^T[128 d x 16]   += V^T[128 d x 128 keys] . P^T[128 x 16] (MN-major A)
// both accumulating in fp32 in TMEM.  Thread t of the four softmax warps owns
// TMEM lane t: key t of S^T, dim t of O^T.
//
// Two CTAs per SM.  A CTA takes 111 KB of shared memory and 192 threads, so
// the next launch's CTAs (the next layer of an engine step) become resident
// beside this launch's as soon as it lets them launch: they plan, allocate
// TMEM and load their first block-table entries while this launch streams,
// and start copying the moment it completes.  K and V tiles share one ring
// of three 32 KiB slots (K of tile t, then V of tile t), a K slot freed as
// soon as its S^T is computed, a V slot when its PV is.
//
// Roles (192 threads): warps 0-3 run the softmax and, at the end of each
// piece, its epilogue (normalise, write the output or a partial piece, merge,
// fold a shared prefix's states); warp 4 plans and issues the TMA copies (it
// plans before the CTA's set-up, and K/V tiles are evict-first in L2: each
// is read once); one thread of warp 5 issues the MMAs.  e4m3 pools add warps
// 6-9 (320 threads), which widen the codes to f16: K tiles into TMEM, V tiles
// into a shared-memory operand; Q and P are then f16 too.  S and O^T are
// double buffered in TMEM, so the MMAs of the next piece proceed while the
// softmax warps finish the previous one.
// The running maximum is raised only when a score exceeds it by more than
// 2^8 (a CTA-wide vote), so the common tile needs no cross-thread reduction;
// O^T is rescaled in TMEM on the rare raise.
#include <climits>

#include "pkv_internal.h"
#include "pkv_plan.cuh"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

using plan::Piece;
using plan::kEndRow;

constexpr int kTcWarps = 6;                 // 0-3 softmax + epilogue, 4 producer, 5 MMA
constexpr int kTcThreads = 32 * kTcWarps;
// e4m3 pools: four more warps (6-9), one per TMEM lane quarter, widen the
// codes to f16 (one hardware conversion per pair of codes): K rows straight
// into TMEM, where the S^T MMA reads its A operand, V rows into a shared-
// memory operand; Q and P are then f16 as well, since both operands of a
// kind::f16 MMA must have the same type.
constexpr int kConvWarps = 4;
constexpr int kTcThreadsF8 = kTcThreads + 32 * kConvWarps;
constexpr int kRawTile = 128 * kHeadDim;   // one 128-key tile of e4m3 codes (bytes)
constexpr int kRawSlots = 4;               // e4m3 ring: K or V codes of one tile
constexpr int kTile = 128;                 // keys per tile (MMA M of S^T, K of PV)
constexpr int kBlkPerTile = kTile / kBlockSize;
constexpr int kN = 16;                     // MMA N: the group's heads, padded
constexpr int kHalf = kTile * 128;         // one 64-dim half of a 128-key bf16 tile
constexpr int kOpHalf = kN * 128;          // one 64-element half of a 16-row operand
constexpr int kSlots = 3;                  // ring slots (32 KiB): K or V of one tile
// TMEM columns: S0 0..15, S1 16..31, O0 32..47, O1 48..63; e4m3 pools also
// hold the widened K tiles there (two buffers of 64 columns: 128 keys x 128 d
// f16, two d per column).
constexpr uint32_t kColO = 32;             // O^T of piece j in columns kColO + (j & 1) * kN
constexpr uint32_t kColK = 64;             // e4m3: K tile t in columns kColK + (t & 1) * 64
constexpr float kNegBig = -1.0e30f;
constexpr float kLazyMargin = 8.f;         // log2 of the largest probability allowed
constexpr int kBarSoftmax = 1;             // named barrier of the four softmax warps
constexpr int kSoftThreads = 128;
constexpr int kPastPiece = INT_MIN;        // block-table slot past the piece (not read)
constexpr int kWindow = 32;                // block-table entries loaded at a time (4 tiles)

// Debug-only per-tile timeline of CTA 0 (build with -DPKV_TC_TRACE=1):
// %globaltimer at load issue, keys seen by the MMA warp, scores seen by the
// softmax, PV issue, and slot release seen by the producer; e4m3 pools also
// K (7) and V (8) widened by the converters.
#ifndef PKV_TC_TRACE
#define PKV_TC_TRACE 0
#endif
#if PKV_TC_TRACE
constexpr int kTrTiles = 64;
__device__ unsigned long long g_tc_trace[9][kTrTiles];
#define TC_TR(ev, tile) do { if (blockIdx.x == 0 && (tile) < kTrTiles) g_tc_trace[ev][tile] = global_timer_ns(); } while (0)
#else
#define TC_TR(ev, tile) do { } while (0)
#endif
// With PKV_TC_TRACE >= 3 also a per-CTA timeline of the whole kernel, one
// set of events per launch (slot chosen by the out pointer): 0 entry, 1
// set-up done, 2 producer ready, 3 first load issued, 4 first keys seen by the
// MMA warp, 5 last PV issued, 6 last piece written, 7 exit, 8 SM id + 1, 9
// grid-dependency wait taken (early_kv), 10 plan done, 11 first pieces
// known, 16 O read from TMEM, 17 last O commit issued.
#if PKV_TC_TRACE >= 3
// Slots by the out pointer, so that consecutive launches keep their own.
constexpr int kTrCtas = 256, kTrSlots = 32;
__device__ unsigned long long g_tc_cta[kTrSlots][kTrCtas][18];
#define TC_CTA(ev) do { if (blockIdx.x < kTrCtas) g_tc_cta[(uint32_t)((reinterpret_cast<uintptr_t>(p.out) >> 8) * 0x9E3779B1u) >> 27][blockIdx.x][ev] = global_timer_ns(); } while (0)
#define TC_CTA_VAL(ev, v) do { if (blockIdx.x < kTrCtas) g_tc_cta[(uint32_t)((reinterpret_cast<uintptr_t>(p.out) >> 8) * 0x9E3779B1u) >> 27][blockIdx.x][ev] = (v); } while (0)
#else
#define TC_CTA(ev) do { } while (0)
#define TC_CTA_VAL(ev, v) do { } while (0)
#endif

struct __align__(1024) TcSmem {
  union {
    // bf16: ring occupant n (n = 0, 1, 2, ...) lives in slot n % kSlots: the
    // K tile of tile n / 2 when n is even, its V tile when n is odd; [d half]
    // 128 keys x 64 d, 128-byte swizzled.
    uint8_t slot[kSlots][2][kHalf];
    struct {
      // e4m3: occupant n's codes in raw slot n % kRawSlots (128 keys x 128
      // codes, 128-byte swizzled), and the widened V operand of one tile.
      uint8_t raw[kRawSlots][kRawTile];
      uint8_t vbuf[2][kHalf];
    } f8;
  };
  uint8_t q[2][2][kOpHalf];       // [piece buffer][d half]: Q rows (heads), rows >= g zero
  uint8_t pt[2][kOpHalf];         // [key half]: P^T as 16 rows (heads) x 64 keys
  float red[4][kN];               // per-warp partial maxima (softmax warps)
  float st_l[4][kN];              // per-warp normaliser partial sums (epilogue)
  Piece pinfo[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t full[kSlots], empty[kSlots];  // bf16: occupant landed / released
  uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];  // e4m3: codes landed / read
  uint64_t kt_full[2], kt_free[2];  // e4m3: K tile widened into TMEM / read by S^T
  uint64_t v_full, v_free;        // e4m3: V operand widened / read by the PV
  uint64_t q_conv[2];             // e4m3 pools: Q buffer converted to f16 by the softmax warps
  uint64_t s_full[2], s_free[2];  // S^T buffer computed / read by the softmax
  uint64_t p_full, p_free;        // P^T written by the softmax / read by the PV
  uint64_t o_full[2], o_empty[2];  // O^T buffer complete / read by the epilogue
  uint64_t mma_done;              // an aborted CTA's last tcgen05.commit
  uint32_t tmem_base;
  WaitCtl wait;                   // abort flag and wait limit of the bounded waits
  int is_last;
  int idle;                       // the plan gave this CTA no work
  int conv_end;                   // e4m3 pools: ring occupants issued in all (set at the end)
  int raw_valid[kRawSlots];       // e4m3: leading rows of the occupant's tile that hold keys
};

__device__ __forceinline__ float warp_max(float v) {
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The spin of a bounded mbarrier wait (mbar_wait) after a first probe that
// failed, out of line: one copy in the kernel instead of one per wait.  The
// bf16 kernel's smaller instruction footprint measured 0.5 us faster per
// launch on a 64 x 512 decode; the e4m3 kernel (96 registers) and the other
// kernels were slower with the call and keep the inline spin.
static __device__ __noinline__ bool tc_wait_spin(uint64_t* bar, uint32_t parity, int* err,
                                                 WaitCtl* ctl) {
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (ctl->abort) return false;
    #pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > ctl->limit_ns) {
      record_error(err, kErrTimeout);
      ctl->abort = 1;
      return false;
    }
  }
}

// mbar_wait, with the spin out of line unless `kInline`.
template <bool kInline>
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, int* err, WaitCtl* ctl) {
  if constexpr (kInline) {
    return mbar_wait(bar, parity, err, ctl);
  } else {
    return mbar_try_wait(bar, parity) || tc_wait_spin(bar, parity, err, ctl);
  }
}

// Shared-prefix (cascade) rows: folds the prefix pass's partial states of
// output dim d of row-head `rh` (row * Hq + head) into (M, num, den) by
// log-sum-exp.  The prefix pass left one partial per chunk of the `shared`
// keys: a normalised output and its (max, normaliser), stride `stride` rows
// apart.  Out of line: only cascade calls reach it, and one copy keeps the
// kernel's instruction footprint small.
struct PrefixFold {
  float M, num, den;
};
static __device__ __noinline__ PrefixFold fold_prefix_states(const float* pre_o,
                                                             const float* pre_ml,
                                                             long long rh, long long stride,
                                                             int shared, int d, PrefixFold f) {
  const int nch = prefix_chunks(shared);
  // all chunks' loads first (they were prefetched into L2), then fold
  float2 ml[kPrefixSplits];
  float ov[kPrefixSplits];
  #pragma unroll
  for (int c = 0; c < kPrefixSplits; ++c) {
    if (c < nch) {
      const long long sl2 = c * stride + rh;
      ml[c] = __ldcg(reinterpret_cast<const float2*>(pre_ml + sl2 * 2));
      ov[c] = __ldcg(pre_o + sl2 * kHeadDim + d);
    }
  }
  #pragma unroll
  for (int c = 0; c < kPrefixSplits; ++c) {
    if (c < nch) {
      const float Mn = fmaxf(f.M, ml[c].x);
      const float a = fast_exp2(f.M - Mn), w = fast_exp2(ml[c].x - Mn) * ml[c].y;
      f.num = f.num * a + w * ov[c];
      f.den = f.den * a + w;
      f.M = Mn;
    }
  }
  return f;
}

// The G heads' states of one output dim: running max, normaliser, output.
struct HeadStates8 {
  float m[8], l[8], o[8];
};

// A shared-prefix row's output (dim d of its G heads; out: the first head's):
// this piece's states folded with the prefix pass's partial states of the
// `shared` keys.  Out of line: cascade calls only.
template <int G>
static __device__ __noinline__ void write_prefixed(const float* pre_o, const float* pre_ml,
                                                   __nv_bfloat16* out, long long rh0,
                                                   long long stride, int shared, int d,
                                                   HeadStates8 st) {
  #pragma unroll
  for (int h = 0; h < G; ++h) {
    const float res = st.l[h] > 0.f ? __fdividef(st.o[h], st.l[h]) : 0.f;
    const PrefixFold f = fold_prefix_states(pre_o, pre_ml, rh0 + h, stride, shared, d,
                                            PrefixFold{st.m[h], st.l[h] * res, st.l[h]});
    out[h * kHeadDim] = __float2bfloat16_rn(f.den > 0.f ? f.num / f.den : 0.f);
  }
}

// The last piece of a split row-group to arrive: merges the pieces' partial
// states of output dim d (each a normalised output and its (max,
// normaliser), in workspace slots 2 (c0 + s) (+1 for piece 0 when odd0)) by
// log-sum-exp, folds the shared prefix's states when `shared` >= 0, and
// writes the G heads' outputs (out: dim d of the row's first head).  Out of
// line: once per row-group, and one copy keeps the instruction footprint
// small.
template <int G>
static __device__ __noinline__ void merge_pieces(const float* ws_ml, const float* ws_o,
                                                 const float* pre_o, const float* pre_ml,
                                                 __nv_bfloat16* out, int c0, int S, int odd0,
                                                 int shared, long long rh0, long long stride,
                                                 int d) {
  PrefixFold f[G];
  #pragma unroll
  for (int h = 0; h < G; ++h) f[h] = PrefixFold{kNegBig, 0.f, 0.f};
  // Piece by piece, the G heads' states loaded together (2G loads in
  // flight: one L2 round trip per piece rather than one per head and piece).
  #pragma unroll 1
  for (int s2 = 0; s2 < S; ++s2) {
    const int slot = 2 * (c0 + s2) + ((s2 == 0 && odd0) ? 1 : 0);
    float2 ml[G];
    float ov[G];
    #pragma unroll
    for (int h = 0; h < G; ++h) {
      const long long sl2 = (long long)slot * G + h;
      ml[h] = __ldcg(reinterpret_cast<const float2*>(ws_ml + sl2 * 2));
      ov[h] = __ldcg(ws_o + sl2 * kHeadDim + d);
    }
    #pragma unroll
    for (int h = 0; h < G; ++h) {
      const float Mn = fmaxf(f[h].M, ml[h].x);
      const float a = fast_exp2(f[h].M - Mn), w = fast_exp2(ml[h].x - Mn) * ml[h].y;
      f[h].num = f[h].num * a + w * ov[h];
      f[h].den = f[h].den * a + w;
      f[h].M = Mn;
    }
  }
  #pragma unroll
  for (int h = 0; h < G; ++h) {
    if (shared >= 0) f[h] = fold_prefix_states(pre_o, pre_ml, rh0 + h, stride, shared, d, f[h]);
    out[h * kHeadDim] = __float2bfloat16_rn(f[h].den > 0.f ? f[h].num / f[h].den : 0.f);
  }
}

// Brings the prefix pass's partial states of the G heads of row-head rh0
// into L2 (G x 512 B of outputs and the (max, normaliser) pairs per chunk of
// the `shared` keys); warp-collective, out of line (cascade calls only).
template <int G>
static __device__ __noinline__ void prefetch_prefix_states(const float* pre_o, const float* pre_ml,
                                                           long long rh0, long long stride,
                                                           int shared, int lane) {
  const int nch = prefix_chunks(shared);
  for (int i = lane; i < nch * (G * 4 + 1); i += 32) {
    const int c = i / (G * 4 + 1), x = i % (G * 4 + 1);
    const char* a = x < G * 4
        ? reinterpret_cast<const char*>(pre_o + ((c * stride + rh0) * kHeadDim)) + x * 128
        : reinterpret_cast<const char*>(pre_ml + (c * stride + rh0) * 2);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  }
}

// O^T's G columns of this thread's TMEM lane (tO) times alpha[h]: the rare
// rescale after a tile raised a running maximum.  Out of line in the e4m3
// kernel (4% faster there; the bf16 kernel was 3% slower with it).
struct Alpha8 {
  float v[8];
};
template <int G>
static __device__ __noinline__ void rescale_ot(uint32_t tO, Alpha8 alpha) {
  tc_fence_after();
  float o[8];
  tmem_ld8(tO, o);
  tc_wait_ld();
  #pragma unroll
  for (int h = 0; h < G; ++h) o[h] *= alpha.v[h];
  tmem_st8(tO, o);
  tc_wait_st();
}

// Key row `row` of a staged bf16 V tile (both 64-dim halves, 128-byte
// swizzled rows) set to zero.  Out of line: it runs only in a request's last
// tile, and only when the request ends inside a block.
static __device__ __noinline__ void zero_v_row(uint8_t* half0, uint8_t* half1, int row) {
  #pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint4* vr = reinterpret_cast<uint4*>((hf ? half1 : half0) + (row >> 3) * 1024 + (row & 7) * 128);
    #pragma unroll
    for (int c = 0; c < 8; ++c) vr[c] = make_uint4(0, 0, 0, 0);
  }
}

// An aborted CTA's producer: waits (bounded) for the copies still in flight
// -- ring occupants n_occ - ring .. n_occ - 1 (barriers full[n % ring]) --
// before the CTA's shared memory is released.  Out of line in the e4m3
// kernel.
static __device__ __noinline__ void drain_ring(uint64_t* full, int ring, int n_occ, int* err,
                                               WaitCtl* ctl) {
  for (int m = max(0, n_occ - ring); m < n_occ; ++m)
    mbar_wait_drain(full + m % ring, (m / ring) & 1, err, ctl);
}

// Two e4m3 codes (low byte first) to two f16 (low half first).  Every e4m3
// value is an f16 value, so the widening (the hardware e4m3x2 -> f16x2
// conversion) is exact.
// Four codes (one 32-bit word, low byte first) become two f16 pairs: codes
// 0, 1 in lo and 2, 3 in hi, one hardware conversion per pair.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Row `row` of a raw e4m3 tile (128 codes, 128-byte swizzle) widened to f16
// in registers: h[8 c8 + i] holds d 16 c8 + 2i, +1 (low half first); a row
// past the request's end (which may hold any code, NaN included) becomes
// zeros, so that 0 * V stays 0.
__device__ __forceinline__ void widen_e4m3_row(const uint8_t* raw, int row, bool zero,
                                               uint32_t (&h)[64]) {
  const int sw = row & 7;
  #pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    const uint4 v = zero ? make_uint4(0, 0, 0, 0) : lds128(raw + row * 128 + ((c8 ^ sw) * 16));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
    for (int j = 0; j < 4; ++j) e4m3x4_to_f16x4(w[j], h[c8 * 8 + 2 * j], h[c8 * 8 + 2 * j + 1]);
  }
}

// The widened row into the V operand: d 0..63 in half0, d 64..127 in half1,
// the same swizzled row layout a bf16 tile has.
__device__ __forceinline__ void store_f16_row(const uint32_t (&h)[64], uint8_t* half0,
                                              uint8_t* half1, int row) {
  const int sw = row & 7;
  #pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    uint8_t* dst = (c8 < 4 ? half0 : half1) + row * 128;
    const int c = (c8 & 3) * 2;
    const uint32_t* b = &h[c8 * 8];
    *reinterpret_cast<uint4*>(dst + ((c ^ sw) * 16)) = make_uint4(b[0], b[1], b[2], b[3]);
    *reinterpret_cast<uint4*>(dst + (((c + 1) ^ sw) * 16)) = make_uint4(b[4], b[5], b[6], b[7]);
  }
}

// F8: the pools hold e4m3 codes (kmap / vmap are maps of bytes); K tiles are
// widened into TMEM and V tiles into shared memory, the key scale joins the
// softmax scale and the value scale multiplies the output.
// Registers: bf16 pools cap them at 152 per thread, so that two CTAs (the
// running launch's and the next's) and one CTA of the KV append (8 warps of
// at most 24 registers) fit an SM's 65,536 together; e4m3 pools (320
// threads) take the two-CTA share, 96.
template <int G, bool F8>
__global__ void __launch_bounds__(F8 ? kTcThreadsF8 : kTcThreads, 2) __maxnreg__(F8 ? 96 : 152)
    decode_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  static_assert(G >= 1 && G <= 8, "group size");
  constexpr int kThreads = F8 ? kTcThreadsF8 : kTcThreads;
  constexpr uint32_t kTmemCols = F8 ? 256 : 64;
  constexpr int kRing = F8 ? kRawSlots : kSlots;  // ring slots (K or V of one tile each)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled operands need 1024-byte aligned shared addresses.
  const uint32_t raw = smem_u32(smem_raw);
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  WaitCtl* abort_flag = &sm.wait;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.num_kv_heads;
  if (tid == 0) TC_CTA(0);
#if PKV_TC_TRACE >= 3
  if (tid == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    TC_CTA_VAL(8, smid + 1);
  }
#endif
  // The producer plans before the CTA's set-up whenever the plan's inputs
  // may be read before the grid-dependency wait: seq_lens, query_start_loc
  // and the block table (early_plan).
  const bool early_plan = p.early_plan || p.early_kv;
  plan::Range rg;
  plan::Walker wk;
  Piece pc, pn;
  bool have = false, have_n = false;
  // Block-table entries, 32 blocks (four tiles, one "window") per load and
  // one per lane: the current piece's first two windows (w0, w1) and the next
  // piece's (n0, n1), loaded a piece ahead and checked only when used, so the
  // producer never waits on the table.
  int ent_w0 = kPastPiece, ent_w1 = kPastPiece, ent_n0 = kPastPiece, ent_n1 = kPastPiece;
  auto raw_entries = [&](const Piece& q, int x0) {
    const int x = x0 + lane;
    return x < q.nblk ? __ldg(p.block_tables + (long long)q.r * p.max_blocks + q.b0 + x)
                      : kPastPiece;
  };
  // The next piece becomes the current one and the one after it is fetched
  // (with its first block-table entries, in flight during the next call).
  auto advance = [&]() {
    pc = pn;
    have = have_n;
    ent_w0 = ent_n0;
    ent_w1 = ent_n1;
    have_n = have && wk.next(p, pn);
    ent_n0 = have_n ? raw_entries(pn, 0) : kPastPiece;
    ent_n1 = have_n && pn.nblk > kWindow ? raw_entries(pn, kWindow) : kPastPiece;
  };
  auto plan_first = [&]() {
    plan::plan_cta(p, lane, rg, wk);
    if (lane == 0) TC_CTA(10);
    // the first piece into pn, then into pc with the second into pn (one
    // copy of the walker's code: the loop is not unrolled)
    have_n = true;
    #pragma unroll 1
    for (int i = 0; i < 2; ++i) advance();
    if (lane == 0) TC_CTA(11);
  };
  // One call site for the plan (its code is large): without early_plan its
  // inputs may belong to the kernel before, so the producer waits first.
  if (warp == 4) {
    if (!early_plan) {
      grid_dependency_wait();
      allow_dependent_launch();
    }
    plan_first();
    // The entries must be in registers before the wait below: a volatile
    // use keeps the compiler from sinking their loads past it.
    asm volatile("" ::"r"(ent_w0), "r"(ent_w1), "r"(ent_n0), "r"(ent_n1));
  }
  // A CTA the plan gives no work leaves at once (after the launch wait, so
  // that this grid never completes before the kernel ahead of it): its SM
  // slot goes to the next launch.
  if (warp == 4 && lane == 0) sm.idle = !have;
  __syncthreads();
  if (sm.idle) {
    grid_dependency_wait();
    allow_dependent_launch();
    return;
  }

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_empty[b], 1);   // tcgen05.commit after the piece's last MMA
      mbar_init(&sm.s_full[b], 1);    // tcgen05.commit after S^T = K Q^T into buffer b
      mbar_init(&sm.s_free[b], 4);    // the softmax warps have read S buffer b
      mbar_init(&sm.q_conv[b], 4);    // e4m3 pools: Q buffer b converted by the softmax warps
      mbar_init(&sm.o_full[b], 1);    // tcgen05.commit after the piece's last PV
      mbar_init(&sm.o_empty[b], 4);   // the epilogue (softmax warps) has read O^T buffer b
    }
    mbar_init(&sm.p_full, 4);         // P^T written by the softmax warps
    mbar_init(&sm.p_free, 1);         // tcgen05.commit after the PV that read P^T
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm.full[s], 1);      // bf16: the TMA transaction count
      mbar_init(&sm.empty[s], 1);     // tcgen05.commit after the MMAs that read the slot
    }
    for (int s = 0; s < kRawSlots; ++s) {
      mbar_init(&sm.raw_full[s], 1);           // e4m3: the TMA transaction count
      mbar_init(&sm.raw_empty[s], kConvWarps); // e4m3: the converter warps have read it
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.kt_full[b], kConvWarps);   // e4m3: K tile widened into TMEM buffer b
      mbar_init(&sm.kt_free[b], 1);            // tcgen05.commit after the S^T that read it
    }
    mbar_init(&sm.v_full, kConvWarps);         // e4m3: V operand widened
    mbar_init(&sm.v_free, 1);                  // tcgen05.commit after the PV that read it
    mbar_init(&sm.mma_done, 1);
    sm.wait.abort = 0;
    sm.wait.limit_ns = p.wait_limit_ns;
    sm.conv_end = INT_MAX;
    fence_barrier_init();
  }
  // Operand rows g..15 (padding heads) stay zero for the whole kernel.
  for (int i = tid; i < (int)(sizeof(sm.q) + sizeof(sm.pt)) / 16; i += kThreads) {
    uint8_t* base = i < (int)sizeof(sm.q) / 16 ? &sm.q[0][0][0] + i * 16
                                               : &sm.pt[0][0] + (i - (int)sizeof(sm.q) / 16) * 16;
    *reinterpret_cast<uint4*>(base) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == 5) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (tid == 0) TC_CTA(1);
  // Consumers wait for the previous kernel on the stream here; the producer
  // builds its plan and loads its first block-table entries first (it reads
  // only seq_lens, query_start_loc and block_tables, which with early_plan
  // set the previous kernel does not write).  Each thread lets the next
  // kernel launch only after its own wait.
  //
  // With early_kv the previous kernel is the append of this step's new
  // tokens: before the wait this kernel reads the lengths, the block table
  // and the K/V tiles without a new token, and the producer waits before the
  // first tile that holds one (and before it blocks on a consumer); the
  // softmax and MMA warps read only what it stages.  If that append lets this
  // grid launch as soon as the append starts (early_q unset), q, out and the
  // workspace may still belong to the kernel before the append: Q copies are
  // then issued after the wait and the epilogue waits before its first write.
  if (!p.early_kv && (warp != 4 || !p.early_plan)) {
    grid_dependency_wait();
    allow_dependent_launch();
  }

  if (warp == 4) {
    // ========================= plan + TMA producer =========================
    bool waited = !p.early_kv;
    if (p.early_plan && !p.early_kv) {
      grid_dependency_wait();
      allow_dependent_launch();
    }
    if (lane == 0) TC_CTA(2);
    const int oob_row = p.num_blocks * Hkv * kBlockSize;  // zero-filled by TMA
    // Every K/V tile is read once per call: evict it from L2 first, so that
    // the small per-step arrays (lengths, tables, q) stay cached.
    const uint64_t pol = l2_policy_evict_first();
    // Q copies of pieces met before the wait (at most the two buffers'),
    // issued once it has been taken.
    int q_pend = 0, q_row0 = 0, q_row1 = 0, q_k0 = 0, q_k1 = 0;
    // Per Q buffer: phases armed so far, and whether the last armed phase's
    // copy was issued (an aborted CTA drains the copies in flight).
    int q_armed[2] = {0, 0};
    bool q_copy[2] = {false, false};
    auto issue_q = [&](int ub, int row, int kh) {
      // Testing only: the first piece's q (buffer 0's first phase) is never
      // loaded, so the waits on it run out and the CTA takes the timeout path.
      if (p.debug_withhold_q && ub == 0 && q_armed[0] == 1) return;
      q_copy[ub] = true;
      if (lane == 0) {
        tma_load_3d(sm.q[ub][0], &qmap, 0, kh * G, row, &sm.q_full[ub]);
        tma_load_3d(sm.q[ub][1], &qmap, 64, kh * G, row, &sm.q_full[ub]);
      }
    };
    auto take_wait = [&]() {
      if (!waited) {
        grid_dependency_wait();  // the append of this step's tokens is complete
        allow_dependent_launch();
        waited = true;
        if (lane == 0) TC_CTA(9);
      }
      if (q_pend & 1) issue_q(0, q_row0, q_k0);
      if (q_pend & 2) issue_q(1, q_row1, q_k1);
      q_pend = 0;
    };
    int j = 0, t = 0;  // piece and tile counters
    int n_occ = 0;     // ring occupants whose copies have been issued
    bool ok = true;
    while (ok && have && !abort_flag->abort) {
      const int k = pc.k;
      const int ntile = plan::cdiv(pc.nblk, kBlkPerTile);
      int ent_cur = ent_w0, ent_nxt = ent_w1;
      int ent_nn = ntile > 8 ? raw_entries(pc, 2 * kWindow) : kPastPiece;
      for (int tt = 0; tt < ntile; ++tt, ++t) {
        if (tt > 0 && (tt & 3) == 0) {
          // next window; the one after it was loaded a window ago: warm it
          ent_cur = ent_nxt;
          ent_nxt = ent_nn;
          ent_nn = tt + 8 < ntile ? raw_entries(pc, (tt + 8) * kBlkPerTile) : kPastPiece;
        }
        // Before blocking on the consumers, or before a tile with a new token.
        if (2 * t + 1 >= kRing || pc.b0 + min(pc.nblk, (tt + 1) * kBlkPerTile) - 1 >= pc.fresh) {
          if (!waited || q_pend) take_wait();
        }
        // bf16: lanes 0..15 each copy one (block, d half) of the tile's K or V.
        // e4m3: lanes 0..7 each copy one block's 16 rows of 128 codes into the
        // slot's second half, where the converter warps widen them.  Blocks
        // past the piece are read at an out-of-range row (zero fill).
        const int bsel = lane & 7, hsel = (lane >> 3) & 1;
        const int phys = __shfl_sync(0xffffffffu, ent_cur, (tt & 3) * kBlkPerTile + bsel);
        int row = oob_row;
        if ((unsigned)phys < (unsigned)p.num_blocks) row = (phys * Hkv + k) * kBlockSize;
        else if (phys != kPastPiece && hsel == 0 && lane < 16) record_error(p.err, kErrBounds);
        if (tt == 0) {
          // Q of this piece ahead of its first K/V tile (its copy is the
          // smallest and the first MMA needs it), once the MMAs of piece j-2
          // are done with its buffer.
          const int ub = j & 1;
          if (j >= 2) {
            // (the launch wait is taken: from the third tile on, 2t + 1 >=
            // kRing holds and the producer took it above)
            if (!tc_wait<F8>(&sm.q_empty[ub], ((j >> 1) - 1) & 1, p.err, abort_flag)) {
              ok = false;
              break;
            }
          }
          if (lane == 0) {
            sm.pinfo[ub] = pc;
            mbar_arrive_expect_tx(&sm.q_full[ub], 2u * 64u * G * 2u);
          }
          ++q_armed[ub];
          q_copy[ub] = false;
          if (waited || p.early_q) {
            issue_q(ub, pc.row, k);
          } else {
            q_pend |= 1 << ub;
            if (ub == 0) {
              q_row0 = pc.row;
              q_k0 = k;
            } else {
              q_row1 = pc.row;
              q_k1 = k;
            }
          }
          // The epilogue will fold the prefix pass's partial states of this
          // row: bring them into L2 now.
          if (pc.pre)
            prefetch_prefix_states<G>(p.pre_o, p.pre_ml,
                                      (long long)pc.row * p.num_q_heads + (long long)k * G,
                                      (long long)p.num_q_tokens * p.num_q_heads,
                                      pc.fb * kBlockSize, lane);
          __syncwarp();
        }
        #pragma unroll 1
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const int n = 2 * t + kv;  // ring occupant: K (kv = 0) or V (kv = 1) of tile t
          const int s = n % kRing;
          uint64_t* rel = F8 ? &sm.raw_empty[s] : &sm.empty[s];
          if (n >= kRing && !tc_wait<F8>(rel, ((n / kRing) - 1) & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0 && kv == 0 && t >= 2) TC_TR(4, t - 2);
          if (lane == 0 && kv == 0) TC_TR(0, t);
          if (lane == 0 && t == 0 && kv == 0) TC_CTA(3);
          if (lane == 0) {
            if (F8) {
              // rows of this tile holding keys before the request's end
              const int key0 = (pc.b0 + tt * kBlkPerTile) * kBlockSize;
              sm.raw_valid[s] = max(0, min(kTile, pc.L - key0));
              mbar_arrive_expect_tx(&sm.raw_full[s], (uint32_t)kRawTile);
            } else {
              mbar_arrive_expect_tx(&sm.full[s], 2u * kHalf);
            }
          }
          __syncwarp();
          const CUtensorMap* map = kv == 0 ? &kmap : &vmap;
          if (F8) {
            if (lane < 8) tma_load_2d(sm.f8.raw[s] + bsel * 2048, map, 0, row, &sm.raw_full[s], pol);
          } else if (lane < 16) {
            tma_load_2d(sm.slot[s][hsel] + bsel * 2048, map, hsel * 64, row, &sm.full[s], pol);
          }
          __syncwarp();
          n_occ = n + 1;
        }
        if (!ok) break;
      }
      ++j;
      advance();
    }
    // The CTA finishes after the previous kernel in any case; Q copies still
    // pending are issued unless the CTA is giving up.
    if (abort_flag->abort) q_pend = 0;
    take_wait();
    if (F8 && ok && !abort_flag->abort) {
      // Tell the converter warps that occupant n_occ does not exist:
      // completing the phase they wait on for it, once its slot's previous
      // occupant is done.
      const int s = n_occ % kRawSlots;
      if (n_occ < kRawSlots ||
          tc_wait<F8>(&sm.raw_empty[s], ((n_occ / kRawSlots) - 1) & 1, p.err, abort_flag)) {
        if (lane == 0) {
          *reinterpret_cast<volatile int*>(&sm.conv_end) = n_occ;
          mbar_arrive(&sm.raw_full[s]);
        }
      }
      __syncwarp();
    }
    if (!abort_flag->abort) {
      // End marker: no more pieces for this CTA.  (An aborted CTA sends none:
      // every wait returns at once, and the buffer's phase may already have
      // its arrival.)
      const int ub = j & 1;
      if (j < 2 || tc_wait<F8>(&sm.q_empty[ub], ((j >> 1) - 1) & 1, p.err, abort_flag)) {
        if (lane == 0) {
          sm.pinfo[ub].row = kEndRow;
          mbar_arrive(&sm.q_full[ub]);
        }
      }
    }
    if (abort_flag->abort) {
      // Copies still in flight must land before the CTA's shared memory is
      // released: the last occupant of each slot and the last Q of each buffer.
      if constexpr (F8) {
        drain_ring(sm.raw_full, kRing, n_occ, p.err, abort_flag);
      } else {
        for (int m = max(0, n_occ - kRing); m < n_occ; ++m)
          mbar_wait_drain(&sm.full[m % kRing], (m / kRing) & 1, p.err, abort_flag);
      }
      for (int ub = 0; ub < 2; ++ub)
        if (q_armed[ub] > 0 && q_copy[ub])
          mbar_wait_drain(&sm.q_full[ub], (q_armed[ub] - 1) & 1, p.err, abort_flag);
    }
  } else if (warp == 5) {
    // ============================ MMA issuer ==============================
    // Tile n: O^T += V^T(n-1) P^T(n-1) first, then S^T(n) = K(n) Q^T into S
    // buffer n&1, so the QK^T of a tile overlaps the softmax of the previous.
    if (lane == 0) {
      constexpr uint32_t kIdescS =
          F8 ? idesc_f16_f32(kTile, kN, 0, 0) : idesc_bf16_f32(kTile, kN, 0, 0);
      constexpr uint32_t kIdescO =
          F8 ? idesc_f16_f32(kHeadDim, kN, 1, 0) : idesc_bf16_f32(kHeadDim, kN, 1, 0);
      int t = 0;
      bool ok = true;
      auto pv = [&](int tt, bool first, int j) {
        const int n = 2 * tt + 1, s = n % kSlots, ob = j & 1;
        const uint32_t tO = tmem + kColO + ob * kN;
        ok = ok && tc_wait<F8>(&sm.p_full, tt & 1, p.err, abort_flag);
        ok = ok && (F8 ? tc_wait<F8>(&sm.v_full, tt & 1, p.err, abort_flag)
                       : tc_wait<F8>(&sm.full[s], (n / kSlots) & 1, p.err, abort_flag));
        // O^T buffer ob was last read by the epilogue of piece j - 2.
        if (first && j >= 2)
          ok = ok && tc_wait<F8>(&sm.o_empty[ob], ((j >> 1) - 1) & 1, p.err, abort_flag);
        if (!ok) return;
        TC_TR(3, tt);
        TC_CTA(5);
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // V^T is MN-major (d contiguous): atoms of 64 d x 8 keys, the two d
          // halves kHalf apart, 8-key groups 1024 bytes apart.
          const uint32_t va = F8 ? smem_u32(sm.f8.vbuf[0]) : smem_u32(sm.slot[s][0]);
          const uint64_t da = smem_desc_sw128(va + kk * 2048, kHalf, 1024);
          const uint64_t db = smem_desc_sw128(smem_u32(sm.pt[kk >> 2]) + (kk & 3) * 32, 16, 1024);
          tc_mma_f16_ss(tO, da, db, kIdescO, !first || kk > 0);
        }
        tc_commit(F8 ? &sm.v_free : &sm.empty[s]);
        tc_commit(&sm.p_free);
#if PKV_TC_TRACE >= 2
        tc_wait<F8>(&sm.p_free, tt & 1, p.err, abort_flag);  // PV completion
        TC_TR(6, tt);
#endif
      };
      for (int j = 0; ok; ++j) {
        const int ub = j & 1;
        if (!tc_wait<F8>(&sm.q_full[ub], (j >> 1) & 1, p.err, abort_flag)) break;
        const Piece pc = sm.pinfo[ub];
        if (pc.row == kEndRow) break;
        // e4m3 pools: Q in f16, like the widened K and V
        if (F8 && !tc_wait<F8>(&sm.q_conv[ub], (j >> 1) & 1, p.err, abort_flag)) break;
        const int ntile = plan::cdiv(pc.nblk, kBlkPerTile);
        tc_fence_after();
        for (int tt = 0; tt < ntile && ok; ++tt, ++t) {
          const int b = t & 1, n = 2 * t, s = n % kSlots;
          // The previous tile's PV first: its V slot is released as soon as
          // its probabilities are ready, not after this tile's keys arrive.
          if (tt >= 1) pv(t - 1, tt == 1, j);
          ok = ok && (F8 ? tc_wait<F8>(&sm.kt_full[t & 1], (t >> 1) & 1, p.err, abort_flag)
                         : tc_wait<F8>(&sm.full[s], (n / kSlots) & 1, p.err, abort_flag));
          TC_TR(1, t);
          if (t == 0) TC_CTA(4);
          if (t >= 2) ok = ok && tc_wait<F8>(&sm.s_free[b], ((t >> 1) - 1) & 1, p.err, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tS = tmem + b * kN;
          #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t db =
                smem_desc_sw128(smem_u32(sm.q[ub][kk >> 2]) + (kk & 3) * 32, 16, 1024);
            if (F8) {
              // A = the widened K tile in TMEM: d 16kk .. 16kk+15 in columns 8kk .. 8kk+7
              tc_mma_f16_ts(tS, tmem + kColK + (t & 1) * 64 + kk * 8, db, kIdescS, kk > 0);
            } else {
              const uint64_t da =
                  smem_desc_sw128(smem_u32(sm.slot[s][kk >> 2]) + (kk & 3) * 32, 16, 1024);
              tc_mma_f16_ss(tS, da, db, kIdescS, kk > 0);
            }
          }
          // the K slot (K buffer) is free once S^T is computed
          tc_commit(F8 ? &sm.kt_free[t & 1] : &sm.empty[s]);
          tc_commit(&sm.s_full[b]);
#if PKV_TC_TRACE >= 2
          tc_wait<F8>(&sm.s_full[b], (t >> 1) & 1, p.err, abort_flag);  // QK completion
          TC_TR(5, t);
#endif
        }
        if (ok) pv(t - 1, ntile == 1, j);  // the piece's last tile
        tc_commit(&sm.o_full[ub]);
        TC_CTA(17);
        tc_commit(&sm.q_empty[ub]);
      }
      if (abort_flag->abort) {
        // The MMAs already issued must finish before TMEM is freed.
        tc_commit(&sm.mma_done);
        mbar_wait_drain(&sm.mma_done, 0, p.err, abort_flag);
      }
    }
    __syncwarp();
  } else if (F8 && warp >= kTcWarps) {
    // ================= e4m3 converters (warps 6-9) =======================
    // Occupant by occupant, in the producer's order: thread r widens key row
    // r of the tile (its warp reaches TMEM lanes 32 (warp % 4) .. +31).  A K
    // tile goes into TMEM buffer t & 1 once the S^T of tile t - 2 has read
    // it; a V tile into the shared-memory operand once the PV of tile t - 1
    // has read it.  The raw slot is released as soon as its codes are read.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // K runs one tile ahead: K(0), then K(t + 1) and V(t) for t = 0, 1, ...,
    // so that the S^T of the next tile never waits behind the widening of a
    // V tile, which itself waits for the PV of the tile before.
    auto convert_k = [&](int t) -> bool {
      const int n = 2 * t, s = n % kRawSlots;
      if (!tc_wait<F8>(&sm.raw_full[s], (n / kRawSlots) & 1, p.err, abort_flag)) return false;
      if (n >= *reinterpret_cast<volatile int*>(&sm.conv_end)) return false;
      if (t >= 2 && !tc_wait<F8>(&sm.kt_free[t & 1], ((t >> 1) - 1) & 1, p.err, abort_flag)) return false;
      tc_fence_after();
      const uint8_t* src = sm.f8.raw[s];
      const uint32_t tk = tmem + lane_off + kColK + (t & 1) * 64;
      #pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // d 64 hh .. 64 hh + 63: columns 32 hh .. +31
        uint32_t w[32];
        #pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int c8 = hh * 4 + c;
          const uint4 v = lds128(src + r * 128 + ((c8 ^ (r & 7)) * 16));
          const uint32_t x[4] = {v.x, v.y, v.z, v.w};
          #pragma unroll
          for (int i = 0; i < 4; ++i) e4m3x4_to_f16x4(x[i], w[c * 8 + 2 * i], w[c * 8 + 2 * i + 1]);
        }
        tmem_st32(tk + hh * 32, *reinterpret_cast<const float(*)[32]>(w));
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.raw_empty[s]);
        mbar_arrive(&sm.kt_full[t & 1]);
      }
      if (r == 0) TC_TR(7, t);
      return true;
    };
    auto convert_v = [&](int t) -> bool {
      const int n = 2 * t + 1, s = n % kRawSlots;
      if (!tc_wait<F8>(&sm.raw_full[s], (n / kRawSlots) & 1, p.err, abort_flag)) return false;
      if (n >= *reinterpret_cast<volatile int*>(&sm.conv_end)) return false;
      // The row is widened into registers while the previous tile's PV may
      // still be reading the V operand, and its raw slot goes back at once;
      // only the stores wait for that PV.
      uint32_t hv[64];
      widen_e4m3_row(sm.f8.raw[s], r, r >= sm.raw_valid[s], hv);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.raw_empty[s]);
      if (t >= 1 && !tc_wait<F8>(&sm.v_free, (t - 1) & 1, p.err, abort_flag)) return false;
      store_f16_row(hv, sm.f8.vbuf[0], sm.f8.vbuf[1], r);
      fence_proxy_async_smem();  // generic-proxy writes, read by the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.v_full);
      if (r == 0) TC_TR(8, t);
      return true;
    };
    if (convert_k(0)) {
      for (int t = 0;; ++t) {
        const bool more = convert_k(t + 1);  // false past the last tile (or on abort)
        if (!convert_v(t) || !more) break;
      }
    }
  } else if (warp < 4) {
    // ================ softmax + epilogue (warps 0-3) ======================
    const int row = tid;  // TMEM lane: key `row` of a tile, dim `row` of O^T
    const int d = tid;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    bool out_ready = !(p.early_kv && !p.early_q);  // out and the workspace may be written
    int t = 0;
    for (int j = 0;; ++j) {
      const int ub = j & 1;
      const bool got = tc_wait<F8>(&sm.q_full[ub], (j >> 1) & 1, p.err, abort_flag);
      const Piece pc = sm.pinfo[ub];
      // Agree before any barrier: a wait that gave up (abort) stops everyone.
      if (barrier_or(kBarSoftmax, kSoftThreads, !got || pc.row == kEndRow)) break;
      if (F8) {
        // Q of this piece to f16 in place (2 x 16 rows x 64 dims: two
        // 16-byte chunks per thread), for the MMA's same-type operands
        #pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint4* qp = reinterpret_cast<uint4*>(&sm.q[ub][0][0]) + tid * 2 + c;
          uint4 v = *qp;
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
          #pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_float2(w[i]);
            const __half2 h2 = __floats2half2_rn(f.x, f.y);
            w[i] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *qp = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.q_conv[ub]);
      }
      bool ok = true;
      const uint32_t tO = tmem + lane_off + kColO + ub * kN;
      const int ntile = plan::cdiv(pc.nblk, kBlkPerTile);
      // e4m3: the key scale of this KV head joins the softmax scale
      const float sl =
          F8 && pc.k >= 0 && pc.k < Hkv ? p.scale_log2 * __ldg(p.k_scale + pc.k) : p.scale_log2;
      float m[G], l[G];
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = kNegBig;
        l[h] = 0.f;
      }
      for (int tt = 0; tt < ntile; ++tt, ++t) {
        const int b = t & 1;
        ok = ok && tc_wait<F8>(&sm.s_full[b], (t >> 1) & 1, p.err, abort_flag);
        if (row == 0) TC_TR(2, t);
        tc_fence_after();
        float s[8];
        tmem_ld8(tmem + lane_off + b * kN, s);
        tc_wait_ld();
        // Key `row` of this tile: block x of the tile, offset row % 16.
        const int x = tt * kBlkPerTile + (row >> 4);
        const int pos = (pc.b0 + x) * kBlockSize + (row & 15);
        const bool valid = ok && x < pc.nblk && pos < pc.limit;
        bool over = false;
        #pragma unroll
        for (int h = 0; h < G; ++h) {
          s[h] = valid ? s[h] * sl : -INFINITY;
          over |= s[h] > m[h] + kLazyMargin;
        }
        // S buffer b has been read: the MMA may overwrite it (tile t + 2).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_free[b]);
        // P^T was last read (and O^T last updated) by the PV of tile t - 1.
        if (t >= 1) ok = ok && tc_wait<F8>(&sm.p_free, (t - 1) & 1, p.err, abort_flag);
        if (barrier_or(kBarSoftmax, kSoftThreads, over)) {
          // Raise the running maxima to this tile's; O^T and l move with them.
          #pragma unroll
          for (int h = 0; h < G; ++h) {
            const float mx = warp_max(s[h]);
            if (lane == 0) sm.red[warp][h] = mx;
          }
          named_barrier(kBarSoftmax, kSoftThreads);
          float alpha[8];
          bool grow = false;
          #pragma unroll
          for (int h = 0; h < G; ++h) {
            const float mx = fmaxf(fmaxf(sm.red[0][h], sm.red[1][h]),
                                   fmaxf(sm.red[2][h], sm.red[3][h]));
            const float mn = fmaxf(m[h], mx);
            alpha[h] = fast_exp2(m[h] - mn);
            grow |= mn != m[h];
            m[h] = mn;
            l[h] *= alpha[h];
          }
          if (tt > 0 && grow) {
            if constexpr (F8) {
              Alpha8 a;
              #pragma unroll
              for (int h = 0; h < 8; ++h) a.v[h] = h < G ? alpha[h] : 1.f;
              rescale_ot<G>(tO, a);
            } else {
              tc_fence_after();
              float o[8];
              tmem_ld8(tO, o);
              tc_wait_ld();
              #pragma unroll
              for (int h = 0; h < G; ++h) o[h] *= alpha[h];
              tmem_st8(tO, o);
              tc_wait_st();
            }
          }
          // sm.red is read by every softmax thread before its next write.
          named_barrier(kBarSoftmax, kSoftThreads);
        }
        // p = exp2(s - m) in bf16; P^T row h holds head h, keys contiguous,
        // 128-byte swizzle.  The normaliser sums the rounded values the MMA
        // will use.
        uint8_t* prow = sm.pt[row >> 6];
        const int kc = (row & 63) >> 3;
        #pragma unroll
        for (int h = 0; h < G; ++h) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(prow + (h >> 3) * 1024 + (h & 7) * 128 +
                                                      ((kc ^ (h & 7)) * 16) + (row & 7) * 2);
          if (F8) {  // f16, the type of the widened V
            const __half ph = __float2half_rn(fast_exp2(s[h] - m[h]));
            l[h] += __half2float(ph);
            *dst = *reinterpret_cast<const uint16_t*>(&ph);
          } else {
            const __nv_bfloat16 pb = __float2bfloat16_rn(fast_exp2(s[h] - m[h]));
            l[h] += __bfloat162float(pb);
            *dst = *reinterpret_cast<const uint16_t*>(&pb);
          }
        }
        // Keys past the request's end inside its last block may hold anything
        // (even NaN): zero those V rows so that 0 * V stays 0 in the MMA.
        if (!F8 && x < pc.nblk && pos >= pc.L) {
          const int n = 2 * t + 1, sv = n % kSlots;
          ok = ok && tc_wait<F8>(&sm.full[sv], (n / kSlots) & 1, p.err, abort_flag);
          zero_v_row(sm.slot[sv][0], sm.slot[sv][1], row);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full);
      }
      // ============ epilogue of the piece (same four warps) ================
      // Thread d reads TMEM lane d: dim d of O^T for the g heads.
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        const float sw = warp_sum(l[h]);
        if (lane == 0) sm.st_l[warp][h] = sw;
      }
      named_barrier(kBarSoftmax, kSoftThreads);
      float lt[8];
      #pragma unroll
      for (int h = 0; h < G; ++h)
        lt[h] = (sm.st_l[0][h] + sm.st_l[1][h]) + (sm.st_l[2][h] + sm.st_l[3][h]);
      const bool okO = ok && tc_wait<F8>(&sm.o_full[ub], (j >> 1) & 1, p.err, abort_flag);
      tc_fence_after();
      float o[8];
      tmem_ld8(tO, o);
      tc_wait_ld();
      if (d == 0) TC_CTA(16);
      if (F8) {  // the value scale of this KV head
        const float vs = pc.k >= 0 && pc.k < Hkv ? __ldg(p.v_scale + pc.k) : 0.f;
        #pragma unroll
        for (int h = 0; h < G; ++h) o[h] *= vs;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.o_empty[ub]);
      if (!out_ready) {
        grid_dependency_wait();  // before writing out or the workspace
        out_ready = true;
      }
      const bool in_range = pc.row >= 0 && pc.row < p.num_q_tokens && pc.k >= 0 &&
                            pc.k < Hkv && pc.nblk >= 1 && pc.S >= 1 && pc.c0 >= 0 &&
                            2 * (pc.c0 + pc.S) <= p.num_slots && pc.slot >= 0 &&
                            pc.slot < p.num_slots;
      const long long out_row = ((long long)pc.row * p.num_q_heads + (long long)pc.k * G) * kHeadDim;
      if (in_range && pc.S == 1) {
        if (!okO) {
        } else if (pc.pre) {
          // Shared-prefix (cascade) row: fold in the prefix pass's partial
          // states (pc.b0 is at least the shared block count, and the row's
          // first piece starts exactly there).
          HeadStates8 st;
          #pragma unroll
          for (int h = 0; h < 8; ++h) {
            st.m[h] = h < G ? m[h] : 0.f;
            st.l[h] = h < G ? lt[h] : 0.f;
            st.o[h] = h < G ? o[h] : 0.f;
          }
          write_prefixed<G>(p.pre_o, p.pre_ml, p.out + out_row + d,
                            (long long)pc.row * p.num_q_heads + (long long)pc.k * G,
                            (long long)p.num_q_tokens * p.num_q_heads, pc.fb * kBlockSize, d, st);
        } else {
          #pragma unroll
          for (int h = 0; h < G; ++h)
            p.out[out_row + h * kHeadDim + d] =
                __float2bfloat16_rn(lt[h] > 0.f ? __fdividef(o[h], lt[h]) : 0.f);
        }
      } else if (in_range) {
        // Partial piece: normalised output and (max, normaliser), then the
        // last piece of the row-group to arrive merges all of them.  Every
        // softmax thread takes this branch (pc is shared), so the barriers
        // below are uniform.
        if (okO) {
          #pragma unroll
          for (int h = 0; h < G; ++h) {
            const long long slot = (long long)pc.slot * G + h;
            p.ws_o[slot * kHeadDim + d] = lt[h] > 0.f ? o[h] * __frcp_rn(lt[h]) : 0.f;
            if (d == 0) *reinterpret_cast<float2*>(p.ws_ml + slot * 2) = make_float2(m[h], lt[h]);
          }
        }
        named_barrier(kBarSoftmax, kSoftThreads);
        if (d == 0) {
          // The ticket: release publishes this piece's state (every softmax
          // thread's writes, ordered before this one by the barrier above);
          // acquire makes the other pieces' visible to the merge below.
          int* cnt = p.ws_cnt + (long long)pc.row * Hkv + pc.k;
          const int old = atom_add_acq_rel_gpu(cnt, 1);
          const int last = (old == pc.S - 1);
          if (last) *cnt = 0;  // every piece has arrived: leave the counter at zero
          sm.is_last = last;
        }
        named_barrier(kBarSoftmax, kSoftThreads);
        if (sm.is_last)
          merge_pieces<G>(p.ws_ml, p.ws_o, p.pre_o, p.pre_ml, p.out + out_row + d, pc.c0, pc.S,
                          pc.odd0, pc.pre ? pc.fb * kBlockSize : -1,
                          (long long)pc.row * p.num_q_heads + (long long)pc.k * G,
                          (long long)p.num_q_tokens * p.num_q_heads, d);
      }
      // sm.st_l and sm.is_last are free again once every thread is here.
      named_barrier(kBarSoftmax, kSoftThreads);
      if (d == 0) TC_CTA(6);
    }
  }
  // Every warp reaches this point (aborts only shorten the loops), so the
  // allocating warp can always free TMEM.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
  if (tid == 0) TC_CTA(7);
}

// Two CTAs per SM: each takes at most half of the SM's 228 KiB of shared
// memory, less the 1 KiB the hardware reserves per CTA.
static_assert(sizeof(TcSmem) + 1024 <= (228 * 1024) / 2 - 1024, "two CTAs per SM");

template <int G, bool F8>
cudaError_t launch_decode_tc_g(const DecodeTcLaunch& L, cudaStream_t stream) {
  const size_t smem = sizeof(TcSmem) + 1024;  // + alignment slack
  static unsigned long long configured = 0;   // bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(decode_tc_kernel<G, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    // Two CTAs per SM need the largest shared-memory carveout.
    e = cudaFuncSetAttribute(decode_tc_kernel<G, F8>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(F8 ? kTcThreadsF8 : kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<G, F8>, L.qmap, L.kmap, L.vmap, L.p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

#if PKV_TC_TRACE
cudaError_t decode_tc_trace(void* host, size_t bytes) {
  // [tile timeline of CTA 0][per-CTA timeline][append kernel's per-block timeline]
  cudaError_t e =
      cudaMemcpyFromSymbol(host, g_tc_trace, bytes < sizeof(g_tc_trace) ? bytes : sizeof(g_tc_trace));
#if PKV_TC_TRACE >= 3
  if (e == cudaSuccess && bytes > sizeof(g_tc_trace)) {
    const size_t rest = bytes - sizeof(g_tc_trace);
    uint8_t* h = static_cast<uint8_t*>(host) + sizeof(g_tc_trace);
    e = cudaMemcpyFromSymbol(h, g_tc_cta, rest < sizeof(g_tc_cta) ? rest : sizeof(g_tc_cta));
    if (e == cudaSuccess && rest > sizeof(g_tc_cta))
      e = append_trace(h + sizeof(g_tc_cta), rest - sizeof(g_tc_cta));
  }
#endif
  return e;
}
#endif

cudaError_t launch_decode_tc(const DecodeTcLaunch& L, int group, cudaStream_t stream) {
  if (L.p.kv_fp8) {
    switch (group) {
      case 4: return launch_decode_tc_g<4, true>(L, stream);
      case 5: return launch_decode_tc_g<5, true>(L, stream);
      case 6: return launch_decode_tc_g<6, true>(L, stream);
      case 7: return launch_decode_tc_g<7, true>(L, stream);
      case 8: return launch_decode_tc_g<8, true>(L, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (group) {
    case 4: return launch_decode_tc_g<4, false>(L, stream);
    case 5: return launch_decode_tc_g<5, false>(L, stream);
    case 6: return launch_decode_tc_g<6, false>(L, stream);
    case 7: return launch_decode_tc_g<7, false>(L, stream);
    case 8: return launch_decode_tc_g<8, false>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
