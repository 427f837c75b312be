// fa_fwd_sm103.cu -- exact attention forward (O and per-row LSE) for GB300, sm_103a.
//
// The method is FlashAttention's: S = scale*Q K^T and P = softmax(S) live only
// on chip, and K/V tiles are merged with a running row max m and running
// exp-sum l ("在线Softmax算法" on the aiqz.cc flash-attention-io-optimization
// article: m_new = max(m, m_ij), r = e^(m - m_new), l_new = r l + sum e^(s-m_new),
// O~_new = r O~ + sum e^(s-m_new) v, O = O~/l; the same merge as §5 of the
// zzszmyf.github.io notes "FlashAttention 原理是什么？为什么又省显存又快").
// The loop order is the one of FlashAttention-2 (§9 of the notes page): each
// CTA owns query tiles and streams the K/V tiles of its (batch, head).  The
// structure follows FlashAttention-3 (§10 there): a TMA producer warp fills
// shared memory while the math warps consume it, and softmax work overlaps
// the tensor-core work.
//
// GB300 design (one persistent CTA per SM, 384 threads in three warpgroups):
//   * a work item is a pair of 128-row query tiles (Q_0, Q_1) of one group over one
//     K/V split; both tiles share every K/V tile that is loaded, halving K/V traffic
//     per flop.  The grid holds one CTA per item; a running CTA takes over CTAs that
//     have not started yet (cluster launch control) and does their items itself, so the
//     SMs pick items up in order as they free, and an item's start and end overlap its
//     neighbours' work instead of costing a CTA launch, set-up and drain each;
//   * warps 8-11 give registers to warps 0-7 (setmaxnreg);
//   * warp 8  -- TMA producer and scheduler: per item Q_0, Q_1 (each once the previous
//                item's last S product of that slot has read its buffer), then K_0, V_0,
//                K_1, V_1, ... into one shared-memory ring gated by landed/released
//                mbarriers, continued from item to item; it asks for the next item a few
//                steps before the end of the current one and publishes it to the others;
//   * warp 9  -- MMA issuer (one thread): S_t = Q_t K_j^T with tcgen05.mma
//                (A and B from shared memory, fp32 accumulator in tensor memory),
//                then O_t += P_t V_j with P_t read from tensor memory; P_t is handed
//                over in two halves (keys 0-63, 64-127) through hardware named
//                barriers (bar.arrive by the tile's softmax warps, bar.sync by this
//                warp), so that the first half's products run while the softmax
//                computes the second.  The next item's S products start right after
//                the current item's last P V products;
//   * warps 8, 10, 11 -- convert each landed V tile to fp16 in place for the P V product;
//   * warps 0-3 / 4-7 -- softmax for tile 0 / tile 1, one row per thread:
//                row max, exp2 with scale*log2(e) folded in, running (m, l),
//                fp16 P written back into tensor memory over S_t, and the
//                correction O_t *= r, which only runs when some row's max grew
//                by more than 2^8 (the rescale is exact for any reference m,
//                because l and O~ share it); epilogue O = O~/l -> bf16 -> a ring
//                slot -> TMA store, LSE = m*scale + ln l.
//   * causal: query tile i visits K/V tiles 0..i only; the mask is applied on
//     the diagonal tile (and on a ragged last tile) only; items are numbered
//     longest first.
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 and O_1 after
// that (d columns each).  P_t overwrites the first 64 columns of S_t (16-bit pairs).
//
// Also here: split-K/V (FlashDecoding) with fa_combine_kernel, launched as a programmatic
// dependent of the split kernel; the decode instance fa_fwd_kernel<D, true>, whose CTA runs
// one group's query rows over two splits as two independent chains; and fa_fwd_host, the
// host-to-host forward whose copies overlap the kernels chunk by chunk.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA raises a
// status bit, waits for its own copies and MMAs in flight, frees its tensor
// memory and returns.  The named-barrier waits of the P hand-off cannot be
// bounded; they cannot hang either, because the softmax warps arrive once per
// step whatever happens, and never before the S tile of that step is complete.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa_common.cuh"

namespace fa {

constexpr int kThreads = 384;  // 3 warpgroups: softmax 0, softmax 1, producer + MMA
constexpr uint32_t kSoftmaxRegs = 216;  // setmaxnreg split of the 384 x 168 launch budget:
constexpr uint32_t kOtherRegs = 72;     //   2 x 128 x 216 + 128 x 72 = 384 x 168
constexpr float kRescaleLog2Threshold = 8.0f;  // skip the O correction unless max grows > 2^8
constexpr int kNoWithhold = -1;                 // the test hook's "load every ring tile"

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;           // 128-byte swizzle atoms along d
  static constexpr int kChunkBytes = 128 * 128;    // 128 rows x 64 bf16
  static constexpr int kTileBytes = 128 * D * 2;   // one 128-row tile of Q, K, V or O
  // One ring of tiles, continued from one work item to the next: an item's K_0, V_0, K_1, V_1,
  // ... in the order the MMA warp consumes and releases them (its tile u is K_{u/2} for even u,
  // V_{u/2} for odd u), then, with one split, a staging slot for the epilogue of each of its
  // query tiles that has K/V tiles to visit (O is written there and stored by TMA; the epilogue
  // releases the slot).  A
  // CTA's ring tile g (counted over all its items) sits in slot g % kSlots.  V tiles are
  // numbered J over all items for their conversion barriers.
  static constexpr int kSlots = D == 128 ? 5 : 12;
  static constexpr int kOffQ = 0;                  // Q_0, Q_1
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffBar = kOffRing + kSlots * kTileBytes;
  static constexpr int kBarQFull = 0;                   // one per query tile slot
  static constexpr int kBarQEmpty = 2;                  // one per slot: its item's last S is complete
  // Landed tiles: with one query tile per slot, K tile i (counted over the CTA's items) on
  // kBarFull + i % kSlots and V tile i on kBarVFull + i % kSlots, so that each barrier's phases
  // are waited for in order by the warps that use them; the decode instance's ring on kBarFull
  // by ring position.
  static constexpr int kBarFull = 4;
  static constexpr int kBarEmpty = kBarFull + kSlots;   // per ring slot: its tile released
  static constexpr int kBarVFull = kBarEmpty + kSlots;
  static constexpr int kBarSFull = kBarVFull + kSlots;  // one per query tile slot
  static constexpr int kBarOFinal = kBarSFull + 2;
  static constexpr int kBarOEmpty = kBarOFinal + 2;     // one per slot: its four softmax warps have read O out
  static constexpr int kBarDrain = kBarOEmpty + 2;
  static constexpr int kBarConv = kBarDrain + 1;        // V tile J converted to fp16: J % kSlots
  static constexpr int kBarXchg = kBarConv + kSlots;    // the two converter warps' tile maxima
  static constexpr int kBarItemFull = kBarXchg + 1;     // the next work item published: 2 entries
  static constexpr int kBarItemEmpty = kBarItemFull + 2;
  static constexpr int kBarClc = kBarItemEmpty + 2;     // a take-over request answered
  static constexpr int kNumBars = kBarClc + 1;
  // misc, 16-byte aligned: tmem base (4 B), abort flag (4 B), two published work items (8 B),
  // the 16-byte take-over response, the converters' first-tile maxima (two items x two warps),
  // the fp16 scale exponent K of V per conversion slot
  static constexpr int kOffMisc = (kOffBar + kNumBars * 8 + 15) / 16 * 16;
  static constexpr int kOffItems = kOffMisc + 8;
  static constexpr int kOffClc = kOffMisc + 16;
  static constexpr int kOffXmax = kOffMisc + 32;
  static constexpr int kOffKScale = kOffMisc + 48;
  // each softmax warp's per-item bookkeeping, parked here during the K/V steps (8 x 8 ints)
  static constexpr int kOffPark = (kOffKScale + 4 * kSlots + 15) / 16 * 16;
  static constexpr int kSmemBytes = kOffPark + 256 + 1024;  // + slack for 1024-B alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S_t at t*128
  static constexpr uint32_t kColO = 256;  // O_t at 256 + t*D
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};


// A "group" is the set of query rows that share one K/V head: the G = Hq / Hkv query
// heads of that K/V head, Nq rows each, contiguous in [B, Hq, Nq, d] (R = G * Nq rows).
// Plain multi-head attention is G = 1, Nq = Nk.
struct Params {
  float* lse;        // [groups * R] final LSE (n_splits == 1)
  void* o_bf16;      // [groups * R, D] bf16 final O (n_splits == 1; plain stores for empty tiles)
  float* o_part;     // [n_splits, groups * R, D] fp32 partial O (n_splits > 1)
  float* lse_part;   // [n_splits, groups * R] partial LSE (n_splits > 1)
  int groups;        // B * Hkv
  int R;             // query rows per group
  int Nq;            // query rows per head
  int Nk;            // keys per head
  int q_offset;      // sequence position of each head's query row 0 (causal): Nk - Nq
  int n_qtiles;      // ceil(R / 128)
  int n_cta_q;       // ceil(n_qtiles / 2)
  int n_kv_tiles;    // ceil(Nk / 128)
  int n_splits;      // K/V splits (FlashDecoding); 1 = write the final O and LSE
  int split_tiles;   // K/V tiles per split
  float scale;
  float scale_log2;  // scale * log2(e)
  int causal;
  unsigned long long timeout_ns;
  int withhold_tile;  // test hook instance only: this ring tile (K_0 = 0, V_0 = 1, ...) is never loaded
  const uint16_t* v_raw;  // V [groups, Nk, D] bf16: read directly only to re-convert a tile at a new scale
};

// 2^k as a float, exactly, for k in [-126, 127]
__device__ __forceinline__ float exp2_int(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }
// floor(log2 x) for x > 0 (128 for inf; -127 for subnormals, which only need a large upward scale)
__device__ __forceinline__ int ilog2_float(float x) { return static_cast<int>((__float_as_uint(x) >> 23) & 0xffu) - 127; }

// Rewrites granules base + lane + 32 i (i < N) of a 16-byte-granule tile in shared memory in
// place from bf16 to fp16, kBatch loads in flight at a time; with kMeasure also returns the
// largest magnitude seen by this lane.
template <int N, int kBatch, bool kMeasure>
__device__ __forceinline__ float convert_granules(const uint32_t tile, const int base, const int lane) {
  static_assert(N % kBatch == 0, "whole batches");
  float mx = 0.f;
#pragma unroll 1
  for (int i0 = 0; i0 < N; i0 += kBatch) {
    uint32_t x[kBatch][4];
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      ptx::ld_shared_v4(tile + (base + lane + 32 * (i0 + b)) * 16, x[b][0], x[b][1], x[b][2], x[b][3]);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(x[b][e] << 16), hi = __uint_as_float(x[b][e] & 0xffff0000u);
        if (kMeasure) mx = ptx::fmax3(mx, fabsf(lo), fabsf(hi));
        x[b][e] = ptx::pack_f16x2(lo, hi);
      }
      ptx::st_shared_v4(tile + (base + lane + 32 * (i0 + b)) * 16, x[b][0], x[b][1], x[b][2], x[b][3]);
    }
  }
  return mx;
}

// Last key position (+1 in tiles) any row of query tile qt may see, causal case.
__device__ __forceinline__ int causal_tile_limit(const Params& p, int qt) {
  const int r0 = qt * 128;
  const int r1 = min(r0 + 127, p.R - 1);
  const int max_pos = (r1 / p.Nq != r0 / p.Nq) ? p.q_offset + p.Nq - 1 : p.q_offset + r1 % p.Nq;
  return max_pos < 0 ? 0 : max_pos / 128 + 1;
}

// K/V tiles [lo, lo + n) a query tile visits in the split starting at tile lo; causal tiles end
// at the last key any of its rows may see.
__device__ __forceinline__ int tiles_visible(const Params& p, int qt, int lo) {
  const int hi0 = min(lo + p.split_tiles, p.n_kv_tiles);
  const int hi = p.causal ? min(hi0, causal_tile_limit(p, qt)) : hi0;
  return hi > lo ? hi - lo : 0;
}

// One work item: a group's pair of query tiles over one K/V split (the CTA's tile slots 0 and
// 1).  kDual: one query tile per group and n_splits > 1 (decoding); the two tile slots then
// take the same query rows over splits 2c and 2c+1: two independent softmax/product chains
// per SM, each with its own K/V tiles in the ring.
struct Item {
  int bh;              // group (batch x K/V head)
  int qt0, qt1;        // query tile of each slot
  int split, split1;   // K/V split of each slot
  int lo0, lo1;        // first K/V tile of each slot's split
  int n0, n1;          // K/V tiles each slot visits
  int nmax;
  bool has1;           // slot 1 holds a query tile
};

// Items are numbered longest first for causal attention with one split (the last query tiles
// see the most K/V tiles), otherwise group-major (the items of one K/V head run together and
// share its K and V in L2).  CTA b starts with item b and takes further items over from CTAs
// not yet started, so the SMs pick items up in this order as they free, as the hardware's own
// CTA scheduler would.
template <bool kDual>
__device__ __forceinline__ Item decode_item(const Params& p, int bid) {
  Item it;
  int split = 0, split1 = 0;
  if constexpr (kDual) {
    const int pairs = (p.n_splits + 1) / 2;
    split = 2 * (bid % pairs);
    split1 = split + 1;
    it.bh = bid / pairs;
    it.qt0 = it.qt1 = 0;
    it.has1 = split1 < p.n_splits;
  } else {
    int cta_q;
    if (p.n_splits == 1 && p.causal) {
      cta_q = p.n_cta_q - 1 - bid / p.groups;
      it.bh = bid % p.groups;
    } else {
      split = bid % p.n_splits;
      const int b = bid / p.n_splits;
      it.bh = b / p.n_cta_q;
      cta_q = b % p.n_cta_q;
    }
    split1 = split;
    it.qt0 = 2 * cta_q;
    it.qt1 = it.qt0 + 1;
    it.has1 = it.qt1 < p.n_qtiles;
  }
  it.split = split;
  it.split1 = split1;
  it.lo0 = split * p.split_tiles;
  it.lo1 = split1 * p.split_tiles;
  it.n0 = tiles_visible(p, it.qt0, it.lo0);
  it.n1 = it.has1 ? tiles_visible(p, it.qt1, it.lo1) : 0;
  it.nmax = max(it.n0, it.n1);
  return it;
}

// A persistent CTA per SM: the grid holds one CTA per work item, and each running CTA takes
// over not-yet-started CTAs (cluster launch control) and does their items itself.  Across
// items every role keeps its place in the shared pipelines: the producer loads the next item's
// Q tiles as soon as the current item's last S products have read them and carries the K/V
// ring on, and the MMA warp starts the next item's S products right after the current item's
// last P V products, while the softmax warps are still in the epilogue.  The next item's first
// P V product (which overwrites O) waits until all eight softmax warps have read O out.
template <int D, bool kDual, bool kHook = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const Params p) {
  using C = Cfg<D>;
  constexpr bool kF16 = !kDual;  // P V in fp16: V tiles converted in shared memory
  constexpr int kReaders = kF16 ? 11 : 9;  // warps that read each published item: MMA, softmax, converters
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  volatile int* items = reinterpret_cast<volatile int*>(smem + C::kOffItems);
  volatile int* kscale = reinterpret_cast<volatile int*>(smem + C::kOffKScale);  // per conversion slot
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the split combine (if any) may be scheduled now; it waits for this grid to complete
  ptx::griddep_launch_dependents();

  if (warp == 8 && lane == 0) {
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar(C::kBarQFull + t), 1);
      ptx::mbar_init(bar(C::kBarQEmpty + t), 1);
      ptx::mbar_init(bar(C::kBarSFull + t), 1);
      ptx::mbar_init(bar(C::kBarOFinal + t), 1);
      ptx::mbar_init(bar(C::kBarItemFull + t), 1);
      ptx::mbar_init(bar(C::kBarItemEmpty + t), kReaders);
      ptx::mbar_init(bar(C::kBarOEmpty + t), 4);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      ptx::mbar_init(bar(C::kBarFull + s), 1);
      ptx::mbar_init(bar(C::kBarVFull + s), 1);
      ptx::mbar_init(bar(C::kBarEmpty + s), 1);
      ptx::mbar_init(bar(C::kBarConv + s), 3);
    }
    ptx::mbar_init(bar(C::kBarDrain), 1);
    ptx::mbar_init(bar(C::kBarXchg), 2);
    ptx::mbar_init(bar(C::kBarClc), 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter w{abort_flag, p.timeout_ns};

  // The item after this CTA's item k, as the producer published it: its number, -1 when there
  // is none, -2 when the wait failed.
  auto next_item = [&](const int k) -> int {
    if constexpr (kDual) return -1;
    const int e = k & 1;
    if (!__all_sync(0xffffffffu, w.wait(bar(C::kBarItemFull + e), (k >> 1) & 1))) return -2;
    const int v = items[e];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(C::kBarItemEmpty + e));
    return v;
  };

  // ---- V conversion for the fp16 P V product.  Each landed V tile is rewritten in place as
  // fp16(v * 2^-K), same size and layout; the MMA warp waits for the tile's conversion barrier,
  // which counts three arrivals.  An item's first V tile is converted by warps 10 and 11 in
  // halves (the producer arrives without work); every later tile by three warps on three SM
  // sub-partitions: the producer (warp 8) a quarter, converting V_{j-1} right after it has
  // issued V_j's copy, warps 10 and 11 three eighths each.  K is the item's: 0 whenever its
  // first V tile's largest |v| lies in [2^-4, 65520) (fp16 then holds every value of that size
  // exactly), else chosen so that it lands in [2^14, 2^15), that tile then converted again from
  // global memory; the epilogue multiplies O by 2^K.  Only the first tile is measured.  A later
  // tile too large for fp16 at that scale turns into infinities, which reach every row of the
  // item's O (p * inf, or 0 * inf for a masked key); the epilogue then sets FA_STATUS_V_RANGE:
  // flagged, never silent.  Each converted tile's K is also left in its conversion slot, where
  // the epilogue reads it after waiting for the item's last tile.
  constexpr int kGranT = C::kTileBytes / 16;  // 16-byte granules per tile
  int v_scale = 0;                            // K of the current item, as each converter knows it
  // an item's first V tile (the CTA's V tile J0, ring tile g): warps 10 and 11 (parts 1, 2), a
  // half each, measured; xk counts the items measured before (maxima exchange phase and buffer)
  // V tile J (counted over the CTA's items) has landed: its barrier's earlier phases were each
  // waited for by these warps (or, for the producer, passed before the tile was issued)
  auto wait_v = [&](const int J) -> bool {
    return __all_sync(0xffffffffu, w.wait(bar(C::kBarVFull + J % C::kSlots), (J / C::kSlots) & 1));
  };
  auto convert_first = [&](const int J0, const int g, const int part, const int xk, const int bh,
                           const int kv_row0) -> bool {
    const int slot = g % C::kSlots;
    if (!wait_v(J0)) return false;
    const uint32_t tile = sbase + C::kOffRing + slot * C::kTileBytes;
    {
      const int g0 = (part - 1) * (kGranT / 2);
      float mx = convert_granules<kGranT / 64, 8, true>(tile, g0, lane);
      volatile float* xmax = reinterpret_cast<volatile float*>(smem + C::kOffXmax) + 2 * (xk & 1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) xmax[part - 1] = mx;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kBarXchg));
      if (!__all_sync(0xffffffffu, w.wait(bar(C::kBarXchg), xk & 1))) return false;
      mx = fmaxf(xmax[0], xmax[1]);
      v_scale = 0;
      if (!(mx < 65520.f) || (mx > 0.f && mx < 0.0625f)) {
        v_scale = min(max(ilog2_float(mx) - 14, -100), 100);
        const float mul = exp2_int(-v_scale);
        const size_t row_base = static_cast<size_t>(bh) * p.Nk;
        for (int q = g0 + lane; q < g0 + kGranT / 2; q += 32) {
          const int r = (q >> 3) & 127, c = q >> 10, g = (q & 7) ^ (r & 7);   // 128-byte swizzle
          uint4 v4 = make_uint4(0u, 0u, 0u, 0u);                               // rows past Nk are zero
          if (kv_row0 + r < p.Nk)
            v4 = __ldg(reinterpret_cast<const uint4*>(p.v_raw + (row_base + kv_row0 + r) * D + c * 64 + g * 8));
          uint32_t y[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            y[e] = ptx::pack_f16x2(__uint_as_float(y[e] << 16) * mul, __uint_as_float(y[e] & 0xffff0000u) * mul);
          ptx::st_shared_v4(tile + q * 16, y[0], y[1], y[2], y[3]);
        }
      }
      if (part == 1 && lane == 0) kscale[J0 % C::kSlots] = v_scale;
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(C::kBarConv + J0 % C::kSlots));
    return true;
  };
  // a later V tile J (ring tile g): the producer (part 0) a quarter, warps 10 and 11 three
  // eighths each
  auto convert_share = [&](const int J, const int g, const int part) -> bool {
    const int slot = g % C::kSlots;
    if (!wait_v(J)) return false;
    const uint32_t tile = sbase + C::kOffRing + slot * C::kTileBytes;
    {
      const int g0 = part == 0 ? 0 : part == 1 ? kGranT / 4 : 5 * kGranT / 8;  // granules [g0, g1)
      const int g1 = part == 0 ? kGranT / 4 : part == 1 ? 5 * kGranT / 8 : kGranT;
      if (v_scale != 0) {  // a scaled item (rare): each value times 2^-K on the way
        const float mul = exp2_int(-v_scale);
        for (int q = g0 + lane; q < g1; q += 32) {
          uint32_t x[4];
          ptx::ld_shared_v4(tile + q * 16, x[0], x[1], x[2], x[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            x[e] = ptx::pack_f16x2(__uint_as_float(x[e] << 16) * mul, __uint_as_float(x[e] & 0xffff0000u) * mul);
          ptx::st_shared_v4(tile + q * 16, x[0], x[1], x[2], x[3]);
        }
      } else if (part == 0) {
        convert_granules<kGranT / 128, 8, false>(tile, g0, lane);
      } else {
        convert_granules<3 * kGranT / 256, (3 * kGranT / 256) % 8 ? 4 : 8, false>(tile, g0, lane);
      }
      if (part == 1 && lane == 0) kscale[J % C::kSlots] = v_scale;
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(C::kBarConv + J % C::kSlots));
    return true;
  };
  // the producer's K for the item whose first V tile is J0: known once that tile is converted
  auto producer_scale = [&](const int J0) -> bool {
    if (!__all_sync(0xffffffffu, w.wait(bar(C::kBarConv + J0 % C::kSlots), (J0 / C::kSlots) & 1))) return false;
    v_scale = kscale[J0 % C::kSlots];
    return true;
  };

  if (warp >= 8) ptx::regs_decrease<kOtherRegs>();
  if (warp == 8) {
    // ================================================================ TMA producer and scheduler
    // Lane 0 issues the copies; the whole warp runs the loops, because with fp16 P V it also
    // converts a quarter of each later V tile (V_{j-1} right after V_j's copy is issued).  Per
    // item: the Q tiles (each after the previous item's last S product of that slot has read
    // its buffer), then the item's ring tiles; a few steps before the end of the ring tiles it
    // asks to take over a CTA not yet started, and after them it publishes that CTA's item
    // (or the end) to the other warps.
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::prefetch_tensormap(&tm_o);
    }
    const uint32_t clc_resp = sbase + C::kOffClc;
    int idx = blockIdx.x;
    int U = 0;                // ring tiles issued before the current item
    int Vc = 0;               // V tiles of the items before the current one
    const bool staged = !kDual && p.n_splits == 1;  // each item ends with two O staging slots
    int qn[2] = {0, 0};       // Q tiles loaded per slot
    int n_req = 0;            // take-over requests issued (one phase of kBarClc each)
    bool more = !kDual;       // a request may still find a CTA not yet started
    bool req_open = false;    // a request whose answer has not been read
    int issued = 0;           // ring tiles issued (the decode instance's ring positions)
    int n_k = 0, n_v = 0;     // K and V tiles issued
    int withheld = -1;        // test hook: the first item's ring tile left out
    bool ok = true;
    auto request = [&]() {
      if (lane == 0) {
        ptx::fence_proxy_async_smem();  // the previous answer has been read through the generic proxy
        ptx::mbar_arrive_expect_tx(bar(C::kBarClc), 16);
        ptx::clc_try_cancel(clc_resp, bar(C::kBarClc));
      }
      __syncwarp();
      ++n_req;
      req_open = true;
    };
    for (int k = 0;; ++k) {
      const Item it = decode_item<kDual>(p, idx);
      const int n_tiles = kDual ? 0 : 2 * it.nmax;
      const int u_req = n_tiles > 8 ? n_tiles - 8 : 0;  // ring tile before which to ask for the next item
      if (more && n_tiles == 0) request();
      if (it.nmax >= 1) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || (t ? it.n1 : it.n0) == 0) continue;
          if (qn[t] > 0 && !__all_sync(0xffffffffu, w.wait(bar(C::kBarQEmpty + t), (qn[t] - 1) & 1))) {
            ok = false;
            continue;
          }
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              ptx::tma_load_3d(sbase + C::kOffQ + t * C::kTileBytes + c * C::kChunkBytes, &tm_q,
                               bar(C::kBarQFull + t), c * 64, (t ? it.qt1 : it.qt0) * 128, it.bh);
          }
          __syncwarp();
          ++qn[t];
        }
        if (!ok) break;
        if constexpr (kDual) {
          if (lane == 0) {
            // ring order = the MMA warp's order: per step j and slot t, V_t(j-1) then K_t(j)
            auto load = [&](int kv_tile, bool is_v) -> bool {
              const int u = issued, slot = u % C::kSlots, use = u / C::kSlots;
              if (use > 0 && !w.wait(bar(C::kBarEmpty + slot), (use - 1) & 1)) return false;
              ptx::mbar_arrive_expect_tx(bar(C::kBarFull + slot), C::kTileBytes);
              for (int c = 0; c < C::kChunks; ++c)
                ptx::tma_load_3d(sbase + C::kOffRing + slot * C::kTileBytes + c * C::kChunkBytes,
                                 is_v ? &tm_v : &tm_k, bar(C::kBarFull + slot), c * 64, kv_tile * 128, it.bh);
              issued = u + 1;
              return true;
            };
            for (int j = 0; ok && j <= it.nmax; ++j)
              for (int t = 0; ok && t < 2; ++t) {
                const int nt = t ? it.n1 : it.n0, lo = t ? it.lo1 : it.lo0;
                if (j >= 1 && j - 1 < nt) ok = load(lo + j - 1, true);
                if (ok && j < nt) ok = load(lo + j, false);
              }
          }
          ok = __all_sync(0xffffffffu, ok);
          issued = __shfl_sync(0xffffffffu, issued, 0);
          if (!ok) break;
        }
        const int J0 = Vc;  // the item's first V tile
        for (int u = 0; u < n_tiles; ++u) {
          if (more && u == u_req) request();
          const int g = U + u, slot = g % C::kSlots, use = g / C::kSlots;
          if (use > 0 && !__all_sync(0xffffffffu, w.wait(bar(C::kBarEmpty + slot), (use - 1) & 1))) {
            ok = false;
            break;
          }
          const bool withhold = kHook && k == 0 && u == p.withhold_tile;
          const int ti = Vc + (u >> 1);  // the CTA's K (even u) or V (odd u) tile number
          const uint32_t full = bar(((u & 1) ? C::kBarVFull : C::kBarFull) + ti % C::kSlots);
          if (lane == 0 && !withhold) {
            ptx::mbar_arrive_expect_tx(full, C::kTileBytes);
            const CUtensorMap* m = (u & 1) ? &tm_v : &tm_k;
            for (int c = 0; c < C::kChunks; ++c)
              ptx::tma_load_3d(sbase + C::kOffRing + slot * C::kTileBytes + c * C::kChunkBytes, m, full, c * 64,
                               (it.lo0 + (u >> 1)) * 128, it.bh);
          }
          if (withhold) withheld = u;  // (first item: K or V tile u / 2)
          __syncwarp();
          issued = g + 1;
          if (u & 1) n_v = ti + 1;
          else n_k = ti + 1;
          // its part of the item's first V tile: none.  Arriving only now, after this slot's
          // previous tile was released, keeps the arrival out of the conversion barrier's
          // previous phase (V tile J0 - kSlots, converted before that release).
          if (kF16 && u == 1 && lane == 0) ptx::mbar_arrive(bar(C::kBarConv + J0 % C::kSlots));
          // its quarter of V_{j-1}, right after issuing V_j (j >= 2: V_{j-1} has long landed)
          if (kF16 && (u & 1) && u >= 5) {
            if (u == 5 && !producer_scale(J0)) {
              ok = false;
              break;
            }
            if (!convert_share(J0 + (u >> 1) - 1, U + u - 2, 0)) {
              ok = false;
              break;
            }
          }
        }
        if (kF16 && ok && it.nmax >= 2) {
          if (it.nmax == 2) ok = producer_scale(J0);
          if (ok) ok = convert_share(J0 + it.nmax - 1, U + n_tiles - 1, 0);
        }
        // the staging slots: nothing to load; each epilogue waits for its slot's previous tile
        // to be released, and releases the slot itself
        const int n_stage = staged ? (it.n0 > 0) + (it.n1 > 0) : 0;
        if (!ok) break;
        U += n_tiles + n_stage;
        Vc += it.nmax;
      }
      if (kDual) break;
      // the item after this one: the CTA this item's request took over, if any
      int next = -1;
      if (req_open) {
        if (!__all_sync(0xffffffffu, w.wait(bar(C::kBarClc), (n_req - 1) & 1))) {
          ok = false;
          break;
        }
        req_open = false;
        more = ptx::clc_query(clc_resp, &next);
        if (!more) next = -1;
      }
      // publish it in entry k & 1, once every reader has taken that entry's previous item
      if (k >= 2 && !__all_sync(0xffffffffu, w.wait(bar(C::kBarItemEmpty + (k & 1)), ((k >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        items[k & 1] = next;
        ptx::mbar_arrive(bar(C::kBarItemFull + (k & 1)));
      }
      __syncwarp();
      if (next < 0) break;
      idx = next;
    }
    if (!ok && lane == 0) {  // let every copy already issued land before the CTA's memory is released
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) w.drain(bar(C::kBarQFull + t), (qn[t] - 1) & 1);
      if constexpr (kDual) {
        for (int g = issued - C::kSlots > 0 ? issued - C::kSlots : 0; g < issued; ++g)
          w.drain(bar(C::kBarFull + g % C::kSlots), (g / C::kSlots) & 1);
      } else {
        for (int i = n_k - C::kSlots > 0 ? n_k - C::kSlots : 0; i < n_k; ++i)
          if (withheld != 2 * i) w.drain(bar(C::kBarFull + i % C::kSlots), (i / C::kSlots) & 1);
        for (int i = n_v - C::kSlots > 0 ? n_v - C::kSlots : 0; i < n_v; ++i)
          if (withheld != 2 * i + 1) w.drain(bar(C::kBarVFull + i % C::kSlots), (i / C::kSlots) & 1);
      }
      if (req_open) w.drain(bar(C::kBarClc), (n_req - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================================================================ MMA issuer
    // The whole warp runs the loop (waits and descriptor arithmetic stay warp-uniform);
    // one elected lane issues each MMA and commit.  Descriptors are formed once: a step
    // along a tile is a constant added to the 16-byte-unit address field.
    constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdescPV = kF16 ? ptx::idesc_f16_f32(128, D, true) : ptx::idesc_bf16_f32(128, D, true);
    // Descriptors are kept as their low 32 bits (address and leading offset); the high half is
    // the same constant for Q, K and V (stride 1024 B, 128-byte swizzle) and joins at the MMA.
    constexpr uint32_t kSlotStep = C::kTileBytes >> 4;
    constexpr uint32_t kDescHi32 = ptx::desc_sw128_hi(1024);
    constexpr uint64_t kDescHi = static_cast<uint64_t>(kDescHi32) << 32;
    const uint32_t desc_q0 = ptx::desc_sw128_lo(sbase + C::kOffQ, 16);
    const uint32_t desc_q1 = desc_q0 + kSlotStep;
    const uint32_t desc_k_ring = ptx::desc_sw128_lo(sbase + C::kOffRing, 16);
    // V: N-contiguous; next 64 d-columns at +16 KB (LBO), next 8 keys at +1 KB (SBO)
    const uint32_t desc_v_ring = ptx::desc_sw128_lo(sbase + C::kOffRing, C::kChunkBytes);
    int idx = blockIdx.x;
    int U = 0;            // ring tiles of the items before the current one
    int Vc = 0;           // V tiles of the items before the current one
    const bool staged = !kDual && p.n_splits == 1;
    // barrier parities and flags, one bit each: bit t the next Q-full phase of slot t, bit 2 + t
    // the next O-empty phase of slot t, bit 4 + t set while slot t's O of an earlier item has
    // not been waited for (every earlier epilogue ends before the next item's first P V product)
    uint32_t ph = 0;
    bool ok = true;
    for (int k = 0;; ++k) {
      const Item it = decode_item<kDual>(p, idx);
      if (it.nmax >= 1) {
        if constexpr (kDual) {
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (ok && (t ? it.n1 : it.n0) > 0) ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarQFull + t), 0));
          ptx::tc_fence_after();
          // each tile slot has K/V tiles of its own, consumed (and released) in ring order
          int u = 0;
          for (int j = 0; ok && j <= it.nmax; ++j) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int nt = t ? it.n1 : it.n0;
              if (j >= 1 && j - 1 < nt) {
                ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarFull + u % C::kSlots), (u / C::kSlots) & 1));
                if (!ok) break;
                ptx::named_barrier(3 + t, 160);  // P_t(j-1) handed over in two halves (see the non-dual loop)
                ptx::named_barrier(5 + t, 160);
                ptx::tc_fence_after();
                const uint32_t dv = desc_v_ring + (u % C::kSlots) * kSlotStep;
                const uint32_t t_o = tmem + C::kColO + t * D;
                const uint32_t t_p = tmem + C::kColS + t * 128;
                if (ptx::elect_one()) {
                  if (j > 1) ptx::mma_ts_i<1>(t_o, t_p, kDescHi | dv, kIdescPV);
                  else ptx::mma_ts_i<0>(t_o, t_p, kDescHi | dv, kIdescPV);
#pragma unroll
                  for (int kk = 1; kk < 8; ++kk) ptx::mma_ts_i<1>(t_o, t_p + kk * 8, kDescHi | (dv + kk * 128), kIdescPV);
                  if (j - 1 == nt - 1) ptx::tc_commit(bar(C::kBarOFinal + t));
                  ptx::tc_commit(bar(C::kBarEmpty + u % C::kSlots));
                }
                __syncwarp();
                ++u;
              }
              if (j < nt) {
                ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarFull + u % C::kSlots), (u / C::kSlots) & 1));
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t dk = desc_k_ring + (u % C::kSlots) * kSlotStep;
                const uint32_t t_s = tmem + C::kColS + t * 128;
                const uint32_t dq = t ? desc_q1 : desc_q0;
                if (ptx::elect_one()) {
                  ptx::mma_ss_i<0>(t_s, kDescHi | dq, kDescHi | dk, kIdescQK);
#pragma unroll
                  for (int kk = 1; kk < D / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * (C::kChunkBytes >> 4) + (kk & 3) * 2;
                    ptx::mma_ss_i<1>(t_s, kDescHi | (dq + o), kDescHi | (dk + o), kIdescQK);
                  }
                  ptx::tc_commit(bar(C::kBarSFull + t));
                  ptx::tc_commit(bar(C::kBarEmpty + u % C::kSlots));
                }
                __syncwarp();
                ++u;
              }
            }
          }
        } else {
          // Step 0: S_t = Q_t K_0^T for each tile slot with K/V tiles, then K_0's release.  The
          // steady steps below carry no per-item checks and advance their slot and barrier
          // indices by increments: this warp feeds the tensor pipe, and its loop has to stay short.
          const int n0 = it.n0, n1 = it.n1, nmax = it.nmax;
          const uint32_t s_k0 = U % C::kSlots;
          ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarFull + Vc % C::kSlots), (Vc / C::kSlots) & 1));
          if (ok) ptx::tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int nt = t ? n1 : n0;
            if (!ok || nt == 0) continue;
            ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarQFull + t), (ph >> t) & 1u));  // Q_t of this item
            if (!ok) break;
            ph ^= 1u << t;
            ptx::tc_fence_after();
            const uint32_t t_s = tmem + C::kColS + t * 128;
            const uint32_t dq = t ? desc_q1 : desc_q0, dk = desc_k_ring + s_k0 * kSlotStep;
            if (ptx::elect_one()) {
              ptx::mma_qk_run<kDescHi32>(t_s, dq, dk, kIdescQK, std::make_integer_sequence<int, D / 16>{});
              ptx::tc_commit(bar(C::kBarSFull + t));
              if (nt == 1) ptx::tc_commit(bar(C::kBarQEmpty + t));  // Q_t's buffer free for the next item
            }
            __syncwarp();
          }
          if (ptx::elect_one()) ptx::tc_commit(bar(C::kBarEmpty + s_k0));
          __syncwarp();
          // the item's first P V products overwrite O: every earlier epilogue has read its O out
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (ok && (ph & (16u << t))) {
              ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarOEmpty + t), (ph >> (2 + t)) & 1u));
              ph ^= (4u << t) | (16u << t);
            }
          // steps j = 1 .. nmax: O_t += P_t V_{j-1}, then S_t = Q_t K_j^T
          // V_{j-1}'s ring slot, and its number (J, counted over the CTA's items) modulo 2 kSlots:
          // barrier J % kSlots, phase parity J / kSlots; K_j is ring slot and number one further
          uint32_t s_v = (U + 1) % C::kSlots, n_v = Vc % (2 * C::kSlots);
          for (int j = 1; ok && j <= nmax; ++j) {
            const uint32_t s_k = s_v + 1 == C::kSlots ? 0 : s_v + 1;
            const uint32_t n_k = n_v + 1 == 2 * C::kSlots ? 0 : n_v + 1;
            // V_{j-1} converted to fp16 in its ring slot (the converters waited for it to land)
            ok = __all_sync(0xffffffffu, w.wait(bar((kF16 ? C::kBarConv : C::kBarVFull) + (n_v % C::kSlots)), n_v >= C::kSlots));
            if (!ok) break;
            bool k_ready = false;  // K_j is waited for only right before its first use
            const uint32_t dk = desc_k_ring + s_k * kSlotStep, dv = desc_v_ring + s_v * kSlotStep;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int nt = t ? n1 : n0;
              if (j - 1 < nt) {
                // O_t += P_t V_{j-1}: P from tensor memory (8 columns per 16 keys), V from the ring.
                // The hand-off is a hardware named barrier (tile t's four softmax warps arrive,
                // this warp waits), which wakes far sooner than an mbarrier wait.  It has no
                // timeout, so the softmax warps arrive once per K/V step whatever happens, and
                // never for a step before its S_t is complete (issued after this warp's wait for
                // the step before).  Across items the same holds: the first wait of an item
                // follows the O-empty waits, which the softmax warps pass only by finishing the
                // previous item.
                // P arrives in two halves, keys 0-63 then 64-127 (barriers 3 + t, 5 + t): the first
                // half's products run while the softmax warps compute the second half.
                const uint32_t t_o = tmem + C::kColO + t * D;
                const uint32_t t_p = tmem + C::kColS + t * 128;
                ptx::named_barrier(3 + t, 160);
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                  if (j > 1) ptx::mma_ts_lo<1, kDescHi32, 0, 0>(t_o, t_p, dv, kIdescPV);
                  else ptx::mma_ts_lo<0, kDescHi32, 0, 0>(t_o, t_p, dv, kIdescPV);
                  ptx::mma_pv_run<kDescHi32, 1>(t_o, t_p, dv, kIdescPV, std::make_integer_sequence<int, 3>{});
                }
                __syncwarp();
                ptx::named_barrier(5 + t, 160);
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                  ptx::mma_pv_run<kDescHi32, 4>(t_o, t_p, dv, kIdescPV, std::make_integer_sequence<int, 4>{});
                  if (j == nt) ptx::tc_commit(bar(C::kBarOFinal + t));
                }
                __syncwarp();
              }
              if (j < nt) {
                if (!k_ready) {
                  ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarFull + (n_k % C::kSlots)), n_k >= C::kSlots));
                  if (!ok) break;
                  ptx::tc_fence_after();
                  k_ready = true;
                }
                // S_t = Q_t K_j^T, both K-major: 16 d-columns per step, +32 B inside a 128-byte
                // swizzle atom, next atom (d >= 64) at +16 KB
                const uint32_t t_s = tmem + C::kColS + t * 128;
                const uint32_t dq = t ? desc_q1 : desc_q0;
                if (ptx::elect_one()) {
                  ptx::mma_qk_run<kDescHi32>(t_s, dq, dk, kIdescQK, std::make_integer_sequence<int, D / 16>{});
                  ptx::tc_commit(bar(C::kBarSFull + t));
                  if (j == nt - 1) ptx::tc_commit(bar(C::kBarQEmpty + t));  // Q_t's buffer free for the next item
                }
                __syncwarp();
              }
            }
            if (!ok) break;
            // release in ring order: V_{j-1}, then K_j
            if (ptx::elect_one()) {
              ptx::tc_commit(bar(C::kBarEmpty + s_v));
              if (j < nmax) ptx::tc_commit(bar(C::kBarEmpty + s_k));
            }
            __syncwarp();
            s_v = s_k + 1 == C::kSlots ? 0 : s_k + 1;
            n_v = n_k;
          }
          U += 2 * it.nmax + (staged ? (it.n0 > 0) + (it.n1 > 0) : 0);
          Vc += it.nmax;
        }
        ph |= (it.n0 > 0 ? 16u : 0u) | (it.n1 > 0 ? 32u : 0u);
      }
      if (!ok) break;
      const int nx = next_item(k);
      if (nx == -2) ok = false;
      if (nx < 0) break;
      idx = nx;
    }
    // every MMA issued by this warp completes before tensor memory is freed
    if (ptx::elect_one()) ptx::tc_commit(bar(C::kBarDrain));
    __syncwarp();
    w.drain(bar(C::kBarDrain), 0);
    __syncwarp();
  } else if (kF16 && warp >= 10) {
    // ================================================================ V converters (two of three)
    int idx = blockIdx.x;
    int U = 0, Vc = 0, xk = 0;  // ring tiles and V tiles of the items before, items measured
    const bool staged = p.n_splits == 1;
    for (int k = 0;; ++k) {
      const Item it = decode_item<kDual>(p, idx);
      if (it.nmax >= 1) {
        if (!convert_first(Vc, U + 1, warp - 9, xk, it.bh, it.lo0 * 128)) break;
        ++xk;
        bool good = true;
        for (int j = 1; good && j < it.nmax; ++j) good = convert_share(Vc + j, U + 2 * j + 1, warp - 9);
        if (!good) break;
        U += 2 * it.nmax + (staged ? (it.n0 > 0) + (it.n1 > 0) : 0);
        Vc += it.nmax;
      }
      const int nx = next_item(k);
      if (nx < 0) break;
      idx = nx;
    }
  } else if (warp < 8) {
    // ================================================================ softmax warpgroups
    ptx::regs_increase<kSoftmaxRegs>();
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS + t * 128;
    const uint32_t t_o = tmem + lane_off + C::kColO + t * D;
    const float c2 = p.scale_log2;
    // d = 128: S_t is read in two halves and P written in four parts, which shortens the
    // softmax's span from S ready to P handed over.  d = 64 keeps one load and two stores:
    // its softmax is bound by instruction issue (half the tensor work per exp), and the extra
    // instructions cost it more than the shorter span wins.
    constexpr bool kSplitS = D == 128;
    int idx = blockIdx.x;
    int U = 0;      // ring tiles of the items before the current one
    int Vc = 0;     // V tiles of the items before the current one
    const bool staged = p.n_splits == 1;  // O leaves through the item's staging slot for this tile
    int n_s = 0;    // S_t tiles taken (phases of S-full)
    int n_o = 0;    // final O_t waited for (phases of O-final)
    // The epilogue's row addresses are derived from the item number again after the K/V steps
    // rather than kept live through them: the steps need every register they can get.
    struct Rows {
      size_t grow;      // row in [B*Hq*Nq]
      int my_split;     // the partials this tile slot writes (n_splits > 1)
      bool row_valid;
      int bh, row0;     // the tile's group and first row within it (the TMA store's coordinates)
    };
    auto rows_of = [&](const int item) -> Rows {
      const Item e = decode_item<kDual>(p, item);
      const int row0 = (t ? e.qt1 : e.qt0) * 128, qrow = row0 + row;
      return Rows{static_cast<size_t>(e.bh) * p.R + qrow, t ? e.split1 : e.split, (t == 0 || e.has1) && qrow < p.R,
                  e.bh, row0};
    };
    // no K/V tile of this split is visible to the tile: the empty result (O = 0, LSE = -inf)
    auto write_empty = [&](const Rows& w_) {
      if (!w_.row_valid) return;
      if (p.n_splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.o_bf16) + w_.grow * D * 2);
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        p.lse[w_.grow] = -INFINITY;
      } else {
        float4* dst = reinterpret_cast<float4*>(p.o_part + (static_cast<size_t>(w_.my_split) * p.groups * p.R + w_.grow) * D);
        for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        p.lse_part[static_cast<size_t>(w_.my_split) * p.groups * p.R + w_.grow] = -INFINITY;
      }
    };
    // row 0's staging slot + 1 whose store has not yet been waited for (kept in this warp's park
    // entry 7, not in a register through the K/V steps)
    volatile int* pend = reinterpret_cast<volatile int*>(smem + C::kOffPark) + warp * 8 + 7;
    if (row == 0) *pend = 0;
    for (int k = 0;; ++k) {
      // the previous item's O store: its staging slot is released once the store has read it,
      // here rather than in the epilogue, before any wait of this item (the producer may need
      // the slot before this tile's next S)
      if (row == 0) {
        const int ps = *pend;
        if (ps) {
          ptx::bulk_wait_read<0>();
          ptx::mbar_arrive(bar(C::kBarEmpty + ps - 1));
          *pend = 0;
        }
      }
      const Item it = decode_item<kDual>(p, idx);
      const int nt = t ? it.n1 : it.n0;
      const int qpos = p.q_offset + ((t ? it.qt1 : it.qt0) * 128 + row) % p.Nq;  // sequence position (causal mask)
      if (it.nmax == 0) {  // an item with no K/V tile at all takes no part in the pipelines
        write_empty(rows_of(idx));
      } else {
        // the ring position after this item; this tile's staging slot (if it has K/V tiles) is
        // the last before it, or the one before that for slot 0 when slot 1 has one too
        const int U_next = U + 2 * it.nmax + (staged ? (it.n0 > 0) + (it.n1 > 0) : 0);
        const int stage_g = U_next - 1 - (t == 0 && it.n1 > 0 ? 1 : 0);
        // The K/V steps hold the whole S row, its exponentials and P in registers, right at the
        // warpgroup's budget: the item's bookkeeping waits in shared memory meanwhile (volatile,
        // so that it is read back rather than kept live).
        volatile int* park = reinterpret_cast<volatile int*>(smem + C::kOffPark) + warp * 8;
        park[0] = idx;
        park[1] = k;
        park[2] = U_next;
        park[3] = Vc;
        park[4] = n_o;
        park[5] = stage_g;
        park[6] = it.nmax;
        float m_run = -INFINITY;  // running max of the raw scores q.k (scale > 0)
        float l_run = 0.f;        // running sum of 2^((s - m_run) * c2)
        float lp_run = 0.f;       // bf16 P only: the same sum over the rounded terms
        // One arrive at the P hand-off barrier per K/V step, whatever happens: the MMA warp waits
        // there without a timeout.  After a failed wait the remaining steps of the item only
        // arrive (the loop after this one), each once S_t of its step is complete, so that no
        // arrival runs ahead into a later step's barrier phase: S_t(j) is issued after the MMA
        // warp's wait for step j-1, and the MMA warp cannot wait for step j before issuing it.
        // That wait ignores the abort flag; once the MMA warp has left its loop it ends at the
        // deadline, and the arrivals stop.  The warp then leaves without reading O out, so the
        // MMA warp's wait for that (before the next item's first P V product) fails too.
        bool ok = true;
        int j = 0;
        for (; j < nt; ++j) {
          ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarSFull + t), n_s & 1));
          if (!ok) break;
          ++n_s;
          ptx::tc_fence_after();
          // mask: keys past the end of the sequence, and keys after the query when causal
          const int col0 = ((t ? it.lo1 : it.lo0) + j) * 128;
          int lim = p.Nk - col0;
          if (p.causal && qpos - col0 + 1 < lim) lim = qpos - col0 + 1;
          float s[128];
          float mx0, mx1, mx2, mx3;
          if constexpr (kSplitS) {
            // S_t in two 64-column halves: the row max of the first runs while the second lands
            uint32_t rb[64];
            {
              uint32_t ra[64];
              ptx::tmem_ld64_nowait(t_s, ra);
              ptx::tmem_wait_ld64(ra);
              ptx::tmem_ld64_nowait(t_s + 64, rb);
#pragma unroll
              for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(ra[i]);
            }
            if (lim < 64) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (c >= lim) s[c] = -INFINITY;
            }
            mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c < 60; c += 8) {
              mx0 = ptx::fmax3(mx0, s[c], s[c + 1]);
              mx1 = ptx::fmax3(mx1, s[c + 2], s[c + 3]);
              mx2 = ptx::fmax3(mx2, s[c + 4], s[c + 5]);
              mx3 = ptx::fmax3(mx3, s[c + 6], s[c + 7]);
            }
            mx0 = ptx::fmax3(mx0, s[60], s[61]);
            mx1 = ptx::fmax3(mx1, s[62], s[63]);
            ptx::tmem_wait_ld64(rb);
#pragma unroll
            for (int i = 0; i < 64; ++i) s[64 + i] = __uint_as_float(rb[i]);
            if (lim < 128) {
#pragma unroll
              for (int c = 64; c < 128; ++c)
                if (c >= lim) s[c] = -INFINITY;
            }
#pragma unroll
            for (int c = 64; c < 128; c += 8) {
              mx0 = ptx::fmax3(mx0, s[c], s[c + 1]);
              mx1 = ptx::fmax3(mx1, s[c + 2], s[c + 3]);
              mx2 = ptx::fmax3(mx2, s[c + 4], s[c + 5]);
              mx3 = ptx::fmax3(mx3, s[c + 6], s[c + 7]);
            }
          } else {
            {
              uint32_t r[128];
              ptx::tmem_ld128(t_s, r);
#pragma unroll
              for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(r[i]);
            }
            if (lim < 128) {
#pragma unroll
              for (int c = 0; c < 128; ++c)
                if (c >= lim) s[c] = -INFINITY;
            }
            mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c < 124; c += 8) {
              mx0 = ptx::fmax3(mx0, s[c], s[c + 1]);
              mx1 = ptx::fmax3(mx1, s[c + 2], s[c + 3]);
              mx2 = ptx::fmax3(mx2, s[c + 4], s[c + 5]);
              mx3 = ptx::fmax3(mx3, s[c + 6], s[c + 7]);
            }
            mx0 = ptx::fmax3(mx0, s[124], s[125]);
            mx1 = ptx::fmax3(mx1, s[126], s[127]);
          }
          const float tile_max = fmaxf(ptx::fmax3(mx0, mx1, mx2), mx3);
          const float m_new = fmaxf(m_run, tile_max);
          // Keep the old reference unless the max grew by more than 2^8: l and O~ share the
          // reference, so O = O~/l is unchanged; only the size of the terms is bounded.
          const bool rescale = (m_new - m_run) * c2 > kRescaleLog2Threshold;
          const float m_ref = rescale ? m_new : m_run;
          const float r_fac = rescale ? ptx::ex2_approx((m_run - m_new) * c2) : 1.f;
          // a row that has seen no unmasked key yet keeps m = -inf: its terms are all 0
          const float neg = m_ref == -INFINITY ? 0.f : -m_ref * c2;
          // P = 2^(s*c2 - m_ref*c2), rounded to fp16 pairs for the P V product (bf16 in the
          // decode instance) and written over the first 64 columns of S_t, a part at a time while
          // the rest is computed (four parts with the split S load, two otherwise, so the last
          // store is short).  l_run sums the fp32 values; O = O~ / l_run.  With bf16 P a second sum
          // over the rounded values (lp_run) normalises O instead, which halves O's error when a few
          // keys dominate; fp16 P is 8x finer and needs no second sum.
          __syncwarp();  // reconverge after the per-row mask before the warp-wide TMEM stores
          const float2 c2v = make_float2(c2, c2), negv = make_float2(neg, neg);
          float2 se[4], sp[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) se[i] = sp[i] = make_float2(0.f, 0.f);
          uint32_t pk[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), c2v, negv);
            const float e0 = ptx::ex2_approx(x.x);
            const float e1 = ptx::ex2_approx(x.y);
            se[i & 3] = __fadd2_rn(se[i & 3], make_float2(e0, e1));
            if constexpr (kF16) {
              pk[i] = ptx::pack_f16x2(e0, e1);
            } else {
              pk[i] = ptx::pack_bf16x2(e0, e1);
              sp[i & 3] = __fadd2_rn(sp[i & 3], make_float2(__uint_as_float(pk[i] << 16),
                                                            __uint_as_float(pk[i] & 0xffff0000u)));
            }
            if constexpr (kSplitS) {
              if ((i & 15) == 15) {  // P_t columns [i-15, i]: keys 2(i-15) to 2i+1
                uint32_t part[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) part[k] = pk[i - 15 + k];
                ptx::tmem_st16(t_s + (i - 15), part);
              }
            } else if (i == 31 || i == 63) {  // P_t columns [0,32) (keys 0-63), then [32,64)
              uint32_t half[32];
#pragma unroll
              for (int k = 0; k < 32; ++k) half[k] = pk[i - 31 + k];
              ptx::tmem_st32(t_s + (i - 31), half);
            }
            if (i == 31) {
              // keys 0-63 of P_t(j) are stored: hand them over, after the correction O~ *= r
              // (PV_t(j-1) has completed: the commit behind S_t(j) covers it; PV_t(j) waits for
              // this arrive), so that their products run while the second half is computed
              if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                  uint32_t r[32];
                  ptx::tmem_ld32(t_o + cc * 32, r);
#pragma unroll
                  for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * r_fac);
                  ptx::tmem_st32(t_o + cc * 32, r);
                }
              }
              ptx::tmem_wait_st();
              ptx::tc_fence_before();
              __syncwarp();
              ptx::named_barrier_arrive(3 + t, 160);
            }
          }
          const float2 se01 = __fadd2_rn(se[0], se[1]), se23 = __fadd2_rn(se[2], se[3]);
          l_run = l_run * r_fac + ((se01.x + se01.y) + (se23.x + se23.y));
          if constexpr (!kF16) {
            const float2 sp01 = __fadd2_rn(sp[0], sp[1]), sp23 = __fadd2_rn(sp[2], sp[3]);
            lp_run = lp_run * r_fac + ((sp01.x + sp01.y) + (sp23.x + sp23.y));
          }
          m_run = m_ref;
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          ptx::named_barrier_arrive(5 + t, 160);  // keys 64-127 of P_t(j) handed over to the MMA warp
        }
        if (!ok) {
          for (; j < nt && w.drain(bar(C::kBarSFull + t), n_s & 1); ++j, ++n_s) {
            ptx::named_barrier_arrive(3 + t, 160);
            ptx::named_barrier_arrive(5 + t, 160);
          }
          break;
        }
        idx = park[0];
        k = park[1];
        const int U_after = park[2];
        Vc = park[3];
        n_o = park[4];
        const int stage_at = park[5];
        const int nmax_item = park[6];
        // ---- epilogue: O = O~ / l, LSE = m*scale + ln l; a row that saw no key gets O = 0 and
        // LSE = -inf.  O~ is read out of tensor memory whole, the O-empty barrier arrived at, and
        // the row written from registers: one split, bf16 O straight to its row; several splits,
        // fp32 partial O and partial LSE to the workspace for the combine.
        const uint32_t stage_slot = stage_at % C::kSlots;
        if (nt == 0) {  // no K/V tile for this tile slot: no O, no staging slot, no barrier
          write_empty(rows_of(idx));
        } else {
          ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarOFinal + t), n_o & 1));
          if (!ok) break;
          ++n_o;
          int k_cur = 0;  // fp16 P: O~ is held at V's scale 2^-k_cur, fixed by the item's first V tile
          if constexpr (kF16) {
            // the wait is for this tile's last conversion, which follows the first; that barrier
            // phase cannot have been reused yet: the next item's P V products wait for this
            // epilogue, so the converters are at most a few V tiles ahead of this tile's last
            const int J = Vc + nt - 1;
            ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarConv + J % C::kSlots), (J / C::kSlots) & 1));
            if (!ok) break;
            k_cur = kscale[J % C::kSlots];
          }
          if (staged) {  // the staging slot (long free: it is waited for here, before O is read out)
            // the slot's previous tile has been released (its release is the latest phase the
            // barrier can have completed: the next is this epilogue's own)
            if (stage_at >= C::kSlots)
              ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarEmpty + stage_slot), ((stage_at / C::kSlots) - 1) & 1));
            if (!ok) break;
          }
          ptx::tc_fence_after();
          // O~ leaves in 32-column chunks (a rolled loop: this runs once per item, and the code
          // of the K/V steps is what must stay in the instruction cache)
          const Rows rw = rows_of(idx);
          const bool have = l_run > 0.f;
          // fp16 P: O~ / l at V's scale 2^-k_cur; bf16 P: O~ / (sum of the rounded terms)
          const float inv_l = have ? (kF16 ? exp2_int(k_cur) / l_run : 1.f / lp_run) : 0.f;
          const float lse_row = have ? m_run * p.scale + logf(l_run) : -INFINITY;
          float2 nonfinite = make_float2(0.f, 0.f);  // fp16 P V: stays 0 unless some O~ value is inf or NaN
          // one split: bf16 O through the item's staging slot for this tile (the tile's 128 rows in
          // 64-column chunks, 128-byte swizzle, the layout a K or V tile has there) and TMA
          // stores (rows past the group's end are clipped).  Each thread owns one row, so direct
          // stores would put 32 rows' partial lines into every store instruction and hold the
          // SM's load/store pipe (and with it every warp's shared-memory and barrier operations)
          // for microseconds.  Several splits: fp32 partial O straight to the workspace.
          const uint32_t stage = sbase + C::kOffRing + stage_slot * C::kTileBytes;
          float4* part = reinterpret_cast<float4*>(p.o_part + (static_cast<size_t>(rw.my_split) * p.groups * p.R + rw.grow) * D);
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            ptx::tmem_ld32(t_o + cc * 32, r);
            if constexpr (kF16) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                nonfinite = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                       make_float2(0.f, 0.f), nonfinite);
            }
            if (staged) {
              const uint32_t chunk_base = stage + (cc >> 1) * C::kChunkBytes + row * 128;
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const int gran = (cc & 1) * 4 + g;  // 16-byte granule within the 128-byte row
                ptx::st_shared_v4(chunk_base + ((gran ^ (row & 7)) << 4),
                                  ptx::pack_bf16x2(__uint_as_float(r[8 * g]) * inv_l, __uint_as_float(r[8 * g + 1]) * inv_l),
                                  ptx::pack_bf16x2(__uint_as_float(r[8 * g + 2]) * inv_l, __uint_as_float(r[8 * g + 3]) * inv_l),
                                  ptx::pack_bf16x2(__uint_as_float(r[8 * g + 4]) * inv_l, __uint_as_float(r[8 * g + 5]) * inv_l),
                                  ptx::pack_bf16x2(__uint_as_float(r[8 * g + 6]) * inv_l, __uint_as_float(r[8 * g + 7]) * inv_l));
              }
            } else if (rw.row_valid) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                part[cc * 8 + i] = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                               __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(C::kBarOEmpty + t));  // O_t may be overwritten now
          if (staged) {
            ptx::fence_proxy_async_smem();
            ptx::named_barrier(1 + t, 128);  // all 128 rows written
            if (row == 0) {  // the stores, and the slot's release once they have read it
              for (int c = 0; c < D / 64; ++c) ptx::tma_store_3d(&tm_o, stage + c * C::kChunkBytes, c * 64, rw.row0, rw.bh);
              ptx::bulk_commit();
              *pend = static_cast<int>(stage_slot) + 1;  // released at the next item's top
            }
            if (rw.row_valid) p.lse[rw.grow] = lse_row;
          } else if (rw.row_valid) {
            p.lse_part[static_cast<size_t>(rw.my_split) * p.groups * p.R + rw.grow] = lse_row;
          }
          if (kF16 && __any_sync(0xffffffffu, rw.row_valid && have && l_run < INFINITY &&
                                                   !(nonfinite.x == 0.f && nonfinite.y == 0.f)) && lane == 0)
            atomicOr(&g_status, FA_STATUS_V_RANGE);  // a V tile fp16 could not hold at the item's scale
        }
        U = U_after;
        Vc += nmax_item;
      }
      const int nx = next_item(k);
      if (nx < 0) break;
      idx = nx;
    }
  }

  if (warp < 8 && (threadIdx.x & 127) == 0) ptx::bulk_wait_all();  // the O stores this thread issued
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ==================================================================== split-K/V combine
// FlashDecoding's merge of K/V-split partials (one warp per query row):
//   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s,
// splits that saw no key (LSE_s = -inf) weigh 0; a row with none at all gets O = 0,
// LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256)
    fa_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                      uint16_t* __restrict__ o, float* __restrict__ lse, int rows, int n_splits) {
  constexpr int E = D / 32;  // elements per lane
  ptx::griddep_wait();  // launched behind the split kernel: its partials are complete and visible
  const int row = static_cast<int>((static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int s = 0; s < n_splits; ++s) m = fmaxf(m, lse_part[static_cast<size_t>(s) * rows + row]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float tot = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float w = expf(lse_part[static_cast<size_t>(s) * rows + row] - m);
      tot += w;
      const float* src = o_part + (static_cast<size_t>(s) * rows + row) * D + lane * E;
      if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
        acc[2] += w * x.z;
        acc[3] += w * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
      }
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint32_t packed[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) packed[e] = ptx::pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  uint16_t* dst = o + static_cast<size_t>(row) * D + lane * E;
  if constexpr (E == 4)
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  else
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  if (lane == 0) lse[row] = tot > 0.f ? m + logf(tot) : -INFINITY;
}

// ==================================================================== host side
namespace {

constexpr int kMaxSplits = 1024;
std::mutex g_dev_mutex;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, -1 wrong arch

// Architecture check and the forward kernels' shared-memory limits, once per device.
int prepare_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_dev_state[dev] == 1) return FA_OK;
  if (g_dev_state[dev] == -1) return FA_ERR_ARCH;
  const int arch = check_arch(dev);
  if (arch != FA_OK) {
    if (arch == FA_ERR_ARCH) g_dev_state[dev] = -1;
    return arch;
  }
  if (cudaFuncSetAttribute(fa_fwd_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(fa_fwd_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(fa_fwd_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(fa_fwd_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(fa_fwd_kernel<64, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(fa_fwd_kernel<128, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128>::kSmemBytes) != cudaSuccess)
    return FA_ERR_CUDA;
  g_dev_state[dev] = 1;
  return FA_OK;
}

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk, d;
  float scale;
  int causal;
  int n_splits;
  void* workspace;
  size_t workspace_bytes;
};

// bytes of workspace for n_splits > 1: fp32 partial O, then partial LSE
size_t workspace_needed(long long rows, int d, int n_splits) {
  if (n_splits <= 1) return 0;
  return align256(static_cast<size_t>(n_splits) * rows * d * 4) + align256(static_cast<size_t>(n_splits) * rows * 4);
}

int validate(const Problem& pr) {
  if (!pr.q || !pr.k || !pr.v || !pr.o || !pr.lse) return FA_ERR_ARG;
  if (pr.B < 1 || pr.Hq < 1 || pr.Hkv < 1 || pr.Nq < 1 || pr.Nk < 1 || (pr.d != 64 && pr.d != 128))
    return FA_ERR_ARG;
  if (pr.Hq % pr.Hkv != 0) return FA_ERR_ARG;
  if (!(pr.scale > 0.f) || !std::isfinite(pr.scale)) return FA_ERR_ARG;
  if (pr.n_splits < 1 || pr.n_splits > kMaxSplits) return FA_ERR_ARG;
  const long long q_rows = static_cast<long long>(pr.B) * pr.Hq * pr.Nq;
  const long long kv_rows = static_cast<long long>(pr.B) * pr.Hkv * pr.Nk;
  if (q_rows > 2147483647LL || kv_rows > 2147483647LL) return FA_ERR_ARG;
  const size_t ws = workspace_needed(q_rows, pr.d, pr.n_splits);
  if (ws > 0 && (!pr.workspace || pr.workspace_bytes < ws || (reinterpret_cast<uintptr_t>(pr.workspace) & 255u)))
    return FA_ERR_ARG;
  for (const void* ptr : {pr.q, pr.k, pr.v, static_cast<const void*>(pr.o), static_cast<const void*>(pr.lse)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_ARG;
  const size_t qb = static_cast<size_t>(q_rows) * pr.d * 2, kb = static_cast<size_t>(kv_rows) * pr.d * 2;
  const size_t lb = static_cast<size_t>(q_rows) * 4;
  const struct { const void* p; size_t n; } in[3] = {{pr.q, qb}, {pr.k, kb}, {pr.v, kb}};
  for (const auto& x : in) {
    if (overlaps(pr.o, qb, x.p, x.n) || overlaps(pr.lse, lb, x.p, x.n)) return FA_ERR_ARG;
    if (ws > 0 && overlaps(pr.workspace, ws, x.p, x.n)) return FA_ERR_ARG;
  }
  if (overlaps(pr.o, qb, pr.lse, lb)) return FA_ERR_ARG;
  if (ws > 0 && (overlaps(pr.workspace, ws, pr.o, qb) || overlaps(pr.workspace, ws, pr.lse, lb))) return FA_ERR_ARG;
  for (const void* ptr : {pr.q, pr.k, pr.v, static_cast<const void*>(pr.o), static_cast<const void*>(pr.lse)})
    if (!is_device_pointer(ptr)) return FA_ERR_ARG;
  if (ws > 0 && !is_device_pointer(pr.workspace)) return FA_ERR_ARG;
  return FA_OK;
}

template <int D>
int launch(const Problem& pr, int withhold_tile, unsigned long long timeout_ns, cudaStream_t stream) {
  const int G = pr.Hq / pr.Hkv;
  const int groups = pr.B * pr.Hkv;
  const int R = G * pr.Nq;  // query rows per K/V head (contiguous in [B, Hq, Nq, d])
  CUtensorMap mq, mk, mv, mo;
  if (!encode_map(&mq, pr.q, groups, R, D) || !encode_map(&mk, pr.k, groups, pr.Nk, D) ||
      !encode_map(&mv, pr.v, groups, pr.Nk, D) || !encode_map(&mo, pr.o, groups, R, D))
    return FA_ERR_LAUNCH;
  Params p{};
  p.lse = pr.lse;
  p.o_bf16 = pr.o;
  p.groups = groups;
  p.R = R;
  p.Nq = pr.Nq;
  p.Nk = pr.Nk;
  p.q_offset = pr.Nk - pr.Nq;  // bottom-right causal alignment (square: 0)
  p.n_qtiles = (R + 127) / 128;
  p.n_cta_q = (p.n_qtiles + 1) / 2;
  p.n_kv_tiles = (pr.Nk + 127) / 128;
  p.n_splits = pr.n_splits;
  p.split_tiles = (p.n_kv_tiles + pr.n_splits - 1) / pr.n_splits;
  const long long rows = static_cast<long long>(groups) * R;
  if (pr.n_splits > 1) {
    uint8_t* ws = static_cast<uint8_t*>(pr.workspace);
    p.o_part = reinterpret_cast<float*>(ws);
    p.lse_part = reinterpret_cast<float*>(ws + align256(static_cast<size_t>(pr.n_splits) * rows * D * 4));
  }
  p.scale = pr.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(pr.scale) * 1.4426950408889634);
  p.causal = pr.causal ? 1 : 0;
  const bool dual = p.n_qtiles == 1 && pr.n_splits > 1;
  p.withhold_tile = withhold_tile;
  p.v_raw = static_cast<const uint16_t*>(pr.v);
  p.timeout_ns = timeout_ns;
  const long long grid = dual ? static_cast<long long>(groups) * ((pr.n_splits + 1) / 2)
                              : static_cast<long long>(groups) * p.n_cta_q * pr.n_splits;
  if (grid > 2147483647LL) return FA_ERR_ARG;
  if (dual)
    fa_fwd_kernel<D, true><<<static_cast<unsigned>(grid), kThreads, Cfg<D>::kSmemBytes, stream>>>(mq, mk, mv, mo, p);
  else if (withhold_tile != kNoWithhold)
    fa_fwd_kernel<D, false, true><<<static_cast<unsigned>(grid), kThreads, Cfg<D>::kSmemBytes, stream>>>(mq, mk, mv, mo, p);
  else
    fa_fwd_kernel<D, false><<<static_cast<unsigned>(grid), kThreads, Cfg<D>::kSmemBytes, stream>>>(mq, mk, mv, mo, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  if (pr.n_splits > 1) {
    const long long blocks = (rows * 32 + 255) / 256;
    // programmatic dependent launch: the combine's CTAs are scheduled while the split kernel
    // runs and start the moment it completes, without a launch gap
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fa_combine_kernel<D>, static_cast<const float*>(p.o_part),
                           static_cast<const float*>(p.lse_part), static_cast<uint16_t*>(pr.o), pr.lse,
                           static_cast<int>(rows), pr.n_splits) != cudaSuccess ||
        cudaGetLastError() != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

int run(const Problem& pr, int withhold_tile, unsigned long long timeout_ns, cudaStream_t stream) {
  int rc = validate(pr);
  if (rc != FA_OK) return rc;
  rc = prepare_device();
  if (rc != FA_OK) return rc;
  return pr.d == 64 ? launch<64>(pr, withhold_tile, timeout_ns, stream) : launch<128>(pr, withhold_tile, timeout_ns, stream);
}

Problem mha(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
            float scale, int causal) {
  return Problem{q, k, v, o, lse, B, H, H, N, N, d, scale, causal, 1, nullptr, 0};
}

// ---- fixed device workspace for callers that cannot allocate (fa_fwd_gqa_static_workspace)
// One array per device that loads this library, held until the process exits.  Host code
// must not use the symbol itself as an address: it is a host-side stand-in.  The device
// address comes from cudaGetSymbolAddress, taken once per device with that device current.
constexpr size_t kStaticWorkspaceBytes = FA_STATIC_WORKSPACE_BYTES;
__device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

void* g_static_workspace_addr[kMaxDevices];  // device address per device, set on first use

int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_static_workspace_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    g_static_workspace_addr[dev] = ptr;
  }
  *out = g_static_workspace_addr[dev];
  return FA_OK;
}

// ---- pipelined host-to-host forward (fa_fwd_host); the pipeline itself is in fa_common.cuh
struct HostBuffers {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
};

int run_host(const HostBuffers& h, const Problem& pr, int groups_per_chunk, cudaStream_t stream) {
  if (pr.n_splits != 1) return FA_ERR_ARG;
  int rc = validate(pr);
  if (rc != FA_OK) return rc;
  if (!h.q || !h.k || !h.v || !h.o || !h.lse || groups_per_chunk < 0) return FA_ERR_ARG;
  const int G = pr.Hq / pr.Hkv, groups = pr.B * pr.Hkv;
  const size_t R = static_cast<size_t>(G) * pr.Nq;
  const size_t row_bytes = static_cast<size_t>(pr.d) * 2;
  const size_t qb = groups * R * row_bytes, kb = static_cast<size_t>(groups) * pr.Nk * row_bytes;
  const size_t lb = groups * R * 4;
  const struct { const void* p; size_t n; } in[3] = {{h.q, qb}, {h.k, kb}, {h.v, kb}};
  for (const auto& x : in)
    if (overlaps(h.o, qb, x.p, x.n) || overlaps(h.lse, lb, x.p, x.n)) return FA_ERR_ARG;
  if (overlaps(h.o, qb, h.lse, lb)) return FA_ERR_ARG;
  for (const void* ptr : {h.q, h.k, h.v, static_cast<const void*>(h.o), static_cast<const void*>(h.lse)})
    if (!is_pinned_host(ptr)) return FA_ERR_ARG;
  rc = prepare_device();
  if (rc != FA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe[dev].mu);
  HostPipe* hp = nullptr;
  rc = host_pipe(dev, &hp);
  if (rc != FA_OK) return rc;
  // chunks of whole K/V groups: contiguous rows of Q, O, LSE (R per group) and K, V (Nk)
  int sizes[kMaxChunks];
  // bytes that cross the link (Q, K, V in; O, LSE out) and the attention's flops (the causal
  // fraction taken as one half)
  const double bytes = 2.0 * qb + 2.0 * kb + lb;
  const double flops = 4.0 * static_cast<double>(pr.B) * pr.Hq * pr.Nq * pr.Nk * pr.d * (pr.causal ? 0.5 : 1.0);
  const int n_chunks = chunk_sizes(groups, groups_per_chunk, bytes, flops / kForwardFlopsPerSec, sizes);
  auto at = [](const void* base, size_t off) { return static_cast<const uint8_t*>(base) + off; };
  auto at_mut = [](void* base, size_t off) { return static_cast<uint8_t*>(base) + off; };
  if (cudaEventRecord(hp->start, stream) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int i = 0; i < kComputeStreams; ++i)
    if (cudaStreamWaitEvent(hp->comp[i], hp->start, 0) != cudaSuccess) return FA_ERR_CUDA;
  for (int c = 0, g0 = 0; c < n_chunks; g0 += sizes[c], ++c) {
    const int ng = sizes[c];
    const size_t q_off = g0 * R * row_bytes, q_len = ng * R * row_bytes;
    const size_t k_off = static_cast<size_t>(g0) * pr.Nk * row_bytes, k_len = static_cast<size_t>(ng) * pr.Nk * row_bytes;
    const size_t l_off = g0 * R * 4, l_len = ng * R * 4;
    if (cudaMemcpyAsync(at_mut(const_cast<void*>(pr.q), q_off), at(h.q, q_off), q_len, cudaMemcpyHostToDevice, hp->in) !=
            cudaSuccess ||
        cudaMemcpyAsync(at_mut(const_cast<void*>(pr.k), k_off), at(h.k, k_off), k_len, cudaMemcpyHostToDevice, hp->in) !=
            cudaSuccess ||
        cudaMemcpyAsync(at_mut(const_cast<void*>(pr.v), k_off), at(h.v, k_off), k_len, cudaMemcpyHostToDevice, hp->in) !=
            cudaSuccess ||
        cudaEventRecord(hp->loaded[c], hp->in) != cudaSuccess)
      return FA_ERR_CUDA;
    cudaStream_t cs = hp->comp[c % kComputeStreams];
    if (cudaStreamWaitEvent(cs, hp->loaded[c], 0) != cudaSuccess) return FA_ERR_CUDA;
    Problem sub = pr;
    sub.q = at(pr.q, q_off);
    sub.k = at(pr.k, k_off);
    sub.v = at(pr.v, k_off);
    sub.o = at_mut(pr.o, q_off);
    sub.lse = reinterpret_cast<float*>(at_mut(pr.lse, l_off));
    sub.B = 1;
    sub.Hq = ng * G;
    sub.Hkv = ng;
    rc = pr.d == 64 ? launch<64>(sub, kNoWithhold, kDefaultTimeoutNs, cs) : launch<128>(sub, kNoWithhold, kDefaultTimeoutNs, cs);
    if (rc != FA_OK) return rc;
    if (cudaEventRecord(hp->computed[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.o, q_off), at(pr.o, q_off), q_len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.lse, l_off), at(pr.lse, l_off), l_len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  if (cudaEventRecord(hp->done, hp->out) != cudaSuccess || cudaStreamWaitEvent(stream, hp->done, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

// status words of the backward (fa_bwd_sm103.cu) and FP8 (fa_fp8_sm103.cu) translation
// units: read, optionally cleared
int bwd_status_word(int clear);
int fp8_status_word(int clear);

}  // namespace fa

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, cudaStream_t stream) {
  return fa::run(fa::mha(q, k, v, o, lse, B, H, N, d, scale, causal), fa::kNoWithhold, fa::kDefaultTimeoutNs, stream);
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
               int Nq, int Nk, int d, float scale, int causal, int n_splits, void* workspace,
               size_t workspace_bytes, cudaStream_t stream) {
  const fa::Problem pr{q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, n_splits, workspace, workspace_bytes};
  return fa::run(pr, fa::kNoWithhold, fa::kDefaultTimeoutNs, stream);
}

size_t fa_fwd_gqa_workspace_bytes(int B, int Hq, int Nq, int d, int n_splits) {
  if (B < 1 || Hq < 1 || Nq < 1 || (d != 64 && d != 128) || n_splits < 1 || n_splits > fa::kMaxSplits) return 0;
  return fa::workspace_needed(static_cast<long long>(B) * Hq * Nq, d, n_splits);
}

int fa_fwd_gqa_static_workspace(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                                int n_splits, cudaStream_t stream) {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (n_splits > 1) {
    const size_t need = fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits);
    if (need == 0) return FA_ERR_ARG;  // sizes fa_fwd_gqa would reject anyway
    if (need > fa::kStaticWorkspaceBytes) return FA_ERR_WORKSPACE_TOO_LARGE;
    // every other argument is checked as fa_fwd_gqa checks it, then the device (so that a
    // device of another architecture gets FA_ERR_ARCH, as from fa_fwd_gqa), and only then is
    // the array's address looked up
    const fa::Problem args{q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, 1, nullptr, 0};
    int rc = fa::validate(args);
    if (rc != FA_OK) return rc;
    rc = fa::prepare_device();
    if (rc != FA_OK) return rc;
    rc = fa::static_workspace(&ws);
    if (rc != FA_OK) return rc;
    ws_bytes = fa::kStaticWorkspaceBytes;
  }
  const fa::Problem pr{q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, n_splits, ws, ws_bytes};
  return fa::run(pr, fa::kNoWithhold, fa::kDefaultTimeoutNs, stream);
}

int fa_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                void* q, void* k, void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                float scale, int causal, int groups_per_chunk, cudaStream_t stream) {
  const fa::Problem pr{q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, 1, nullptr, 0};
  return fa::run_host(fa::HostBuffers{q_host, k_host, v_host, o_host, lse_host}, pr, groups_per_chunk, stream);
}

int fa_fwd_withheld_tile(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int N, int d, float scale, int causal, double wait_timeout_ms,
                         cudaStream_t stream) {
  return fa_fwd_withheld_ring_tile(q, k, v, o, lse, B, H, N, d, scale, causal, 1, wait_timeout_ms, stream);
}

int fa_fwd_withheld_ring_tile(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int N, int d, float scale, int causal, int ring_tile, double wait_timeout_ms,
                              cudaStream_t stream) {
  if (!(wait_timeout_ms >= 1.0 && wait_timeout_ms <= 10000.0) || ring_tile < 0) return FA_ERR_ARG;
  return fa::run(fa::mha(q, k, v, o, lse, B, H, N, d, scale, causal), ring_tile,
                 static_cast<unsigned long long>(wait_timeout_ms * 1e6), stream);
}

int fa_status(int clear, cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_status, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  const int bwd_word = fa::bwd_status_word(clear);  // the other translation units' words
  if (bwd_word < 0) return bwd_word;
  const int fp8_word = fa::fp8_status_word(clear);
  if (fp8_word < 0) return fp8_word;
  return static_cast<int>((word | static_cast<unsigned int>(bwd_word) | static_cast<unsigned int>(fp8_word)) &
                          0x7fffffffu);
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_ARG: return "invalid argument (pointer, alignment, size, d, scale, heads or workspace)";
    case FA_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case FA_ERR_LAUNCH: return "kernel launch or TMA descriptor encoding failed";
    case FA_ERR_TIMEOUT: return "a device-side barrier wait timed out";
    case FA_ERR_CUDA: return "CUDA runtime call failed";
    case FA_ERR_WORKSPACE_TOO_LARGE: return "the split-K/V partials need more than the library's fixed workspace";
    default: return "unknown error";
  }
}

int fa_version(void) { return 3; }

}  // extern "C"
