// fa_fp8_sm103.cu -- exact attention forward with FP8 (E4M3) tensor-core products, GB300, sm_103a.
//
// The FP8 forward of §10 item ③ and §12.2 of the zzszmyf.github.io notes "FlashAttention
// 原理是什么？为什么又省显存又快": block-wise quantisation (one scale per block, steadier
// than one per tensor) and incoherent processing (a rotation that spreads the outliers of Q
// and K over all coordinates before they are rounded to FP8).  Here:
//   * q' = (q * sigma) H / sqrt(d) and k' = (k * sigma) H / sqrt(d) per row, H the d x d
//     Hadamard matrix and sigma the caller's random signs: q'.k' = q.k, the scores are
//     unchanged; V is not rotated;
//   * Q', K' and V are cut into 128-row tiles per (batch, head); each tile has one fp32
//     scale s = max|x| / 448 and E4M3 codes e4m3(x / s) (round to nearest even, saturating);
//   * S = (Q'8 K'8^T) s_q s_k from an E4M3 tcgen05 product with fp32 accumulation; the
//     softmax is the forward's online softmax on the true scores;
//   * P is rounded to E4M3 for its product with V as P8 = e4m3(p * 64 * s_v,j / max_t s_v,t)
//     (the factors are folded into the exp2 argument), and O = O~ * max_t s_v,t / (64 l).
//     The rescale threshold is 2^2, so p <= 4 and P8 <= 256 stays inside E4M3's range.
//
// Two kernels on the caller's stream:
//   fa_fp8_prep_kernel -- persistent, two CTAs per SM: the rotation of every 128-row tile of Q
//                         and K as one bf16 tensor-core product with the 128 x 128 rotation
//                         matrix, and the tile maximum, scale and E4M3 codes of Q', K' and V;
//                         V is written transposed (d rows x keys), the K-major layout of its
//                         product with P;
//   fa_fp8_fwd_kernel  -- the bf16 forward's structure (two 128-row query tiles per CTA; a
//                         TMA producer warp; an MMA warp; two softmax warpgroups) with
//                         16 KB E4M3 tiles, a 10-slot K/V ring and kind::f8f6f4 MMAs.
// d = 128, one head per K/V head, queries and keys of the same length, no split.
#include "fa_common.cuh"

namespace fa {

constexpr int kFp8D = 128;
constexpr int kFp8Threads = 384;
constexpr uint32_t kFp8SoftmaxRegs = 216;
constexpr uint32_t kFp8OtherRegs = 72;
constexpr float kFp8RescaleLog2Threshold = 2.0f;  // p <= 4 before the gain of 64
constexpr float kFp8PGainLog2 = 6.0f;              // P8 = e4m3(p * 2^6 * s_v,j / s_v,max)
constexpr int kFp8MaxKvTiles = 1024;              // N <= 131072

// ==================================================================== quantisation
struct QuantParams {
  float* scales[3];        // [BH, n_tiles]
  const int8_t* signs;     // [128], negative = -1
  int BH, N, n_tiles, n_pad;
  unsigned long long timeout_ns;
};

// ==================================================================== preparation
// One persistent kernel prepares all three tensors.  The rotation of a Q or K tile,
// X' = (X * sigma) H / sqrt(128), is the product X R^T with the fixed 128 x 128 matrix
// R[c][k] = sigma_k (-1)^popcount(c & k) (H is symmetric).  R's entries are +-1, exact in bf16,
// so one bf16 tcgen05 product with fp32 accumulation gives the rotation up to the fp32 sums.
// Work items are the 128-row tiles of Q, then of K, then of V, over all heads; CTA b takes
// items b, b + grid, ...  One CTA per SM:
//   warp 0    -- TMA producer: each item's bf16 tile into a four-stage ring;
//   warp 1    -- MMA issuer: per Q or K item one 128 x 128 x 128 product X R^T into one of four
//                tensor-memory accumulators (128 columns each), so that the epilogues of
//                earlier tiles overlap the products of later ones;
//   warps 2-9 -- epilogue in two warpgroups, which take the CTA's even and odd items; one row
//                (Q, K) or one column (V) per thread: the tile maximum, the scale and the E4M3
//                codes.  The codes go to shared memory (each group has two 16 KB buffers, in
//                the 128-byte swizzle) and leave by TMA store, a whole tile at a time.  Q and K codes are (X R^T) * 448 / max|X R^T|: the
//                1/sqrt(128) cancels in the codes and enters the scale only.  V is read from
//                the ring column by column and written transposed (d rows x keys).
// R is built once per CTA in shared memory, in the 128-byte-swizzled K-major layout that the
// product reads.
constexpr int kPrepThreads = 320;
constexpr int kPrepStages = 4;
constexpr int kPrepChunk = 128 * 128;           // 128 rows x 64 bf16 (one swizzle atom wide)
constexpr int kPrepTile = 2 * kPrepChunk;       // one bf16 128 x 128 tile
constexpr int kPrepOffR = 0;
constexpr int kPrepOffRing = kPrepTile;
constexpr int kPrepOffStage = kPrepOffRing + kPrepStages * kPrepTile;  // [group][buffer] 16 KB code tiles
constexpr int kPrepSmemBytes = kPrepOffStage + 4 * 128 * 128 + 1024;   // + slack for 1024-B alignment
constexpr uint32_t kPrepTmemCols = 512;  // four 128-column accumulators

struct PrepBars {
  uint64_t full[kPrepStages], empty[kPrepStages], acc_full[4], acc_empty[4], drain;
};

__global__ void __launch_bounds__(kPrepThreads, 1) fa_fp8_prep_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                       const __grid_constant__ CUtensorMap tm_k,
                                                                       const __grid_constant__ CUtensorMap tm_v,
                                                                       const __grid_constant__ CUtensorMap tm_q8,
                                                                       const __grid_constant__ CUtensorMap tm_k8,
                                                                       const __grid_constant__ CUtensorMap tm_vt8,
                                                                       const QuantParams p) {
  extern __shared__ uint8_t psm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  __shared__ PrepBars bars;
  __shared__ uint32_t tmem_slot, abort_flag;
  __shared__ float warp_max[2][2][4];  // [epilogue group][item parity][warp]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = p.BH * p.n_tiles;  // items per tensor
  const int n_items = 3 * per;
  auto ba = [](uint64_t& x) { return ptx::smem_addr(&x); };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPrepStages; ++i) {
      ptx::mbar_init(ba(bars.full[i]), 1);
      ptx::mbar_init(ba(bars.empty[i]), 1);  // the MMA's commit (Q, K) or one epilogue thread (V)
    }
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(ba(bars.acc_full[i]), 1);
      ptx::mbar_init(ba(bars.acc_empty[i]), 4);  // one arrive per warp of the epilogue group
    }
    ptx::mbar_init(ba(bars.drain), 1);
    abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&tmem_slot), kPrepTmemCols);
    ptx::tmem_relinquish();
  }
  // R: chunk ch holds columns k = 64 ch .. 64 ch + 63 of every row c; 16-byte granule g of a
  // row holds k = 64 ch + 8 g .. + 7 and sits at position g ^ (c mod 8)
  for (int gi = threadIdx.x; gi < 2 * 128 * 8; gi += kPrepThreads) {
    const int ch = gi >> 10, c = (gi >> 3) & 127, g = gi & 7;
    const int k0 = ch * 64 + g * 8;
    uint32_t wd[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int ka = k0 + 2 * e, kb = ka + 1;
      const bool na = (p.signs[ka] < 0) != ((__popc(c & ka) & 1) != 0);
      const bool nb = (p.signs[kb] < 0) != ((__popc(c & kb) & 1) != 0);
      wd[e] = (na ? 0xBF80u : 0x3F80u) | ((nb ? 0xBF80u : 0x3F80u) << 16);  // bf16 -1.0 / +1.0
    }
    ptx::st_shared_v4(sbase + kPrepOffR + ch * kPrepChunk + c * 128 + ((g ^ (c & 7)) << 4), wd[0], wd[1], wd[2],
                      wd[3]);
  }
  ptx::fence_proxy_async_smem();  // R is read by the tensor core (async proxy)
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const Waiter w{&abort_flag, p.timeout_ns};

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      int k = 0, issued = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++k) {
        const int s = k % kPrepStages, use = k / kPrepStages;
        if (use > 0 && !w.wait(ba(bars.empty[s]), (use - 1) & 1)) { ok = false; break; }
        const int which = it / per, rem = it - which * per;
        const int bh = rem / p.n_tiles, tile = rem - bh * p.n_tiles;
        const CUtensorMap* m = which == 0 ? &tm_q : (which == 1 ? &tm_k : &tm_v);
        ptx::mbar_arrive_expect_tx(ba(bars.full[s]), kPrepTile);
        for (int c = 0; c < 2; ++c)  // rows past N arrive as zeros
          ptx::tma_load_3d(sbase + kPrepOffRing + s * kPrepTile + c * kPrepChunk, m, ba(bars.full[s]), c * 64,
                           tile * 128, bh);
        issued = k + 1;
      }
      if (!ok)  // let the copies in flight land before the CTA's memory is released
        for (int kk = issued > kPrepStages ? issued - kPrepStages : 0; kk < issued; ++kk)
          w.drain(ba(bars.full[kk % kPrepStages]), (kk / kPrepStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 128, false);
    const uint64_t db = ptx::smem_desc_sw128(sbase + kPrepOffR, 16, 1024);
    const uint64_t da0 = ptx::smem_desc_sw128(sbase + kPrepOffRing, 16, 1024);
    // Q and K items come first in every CTA's list, so the k-th item is the k-th product;
    // accumulator k mod 4 belongs to epilogue group k mod 2
    int k = 0;
    for (int it = blockIdx.x; it < 2 * per; it += gridDim.x, ++k) {
      const int s = k % kPrepStages, buf = k & 3;
      bool ok = __all_sync(0xffffffffu, w.wait(ba(bars.full[s]), (k / kPrepStages) & 1));
      if (ok && k >= 4) ok = __all_sync(0xffffffffu, w.wait(ba(bars.acc_empty[buf]), ((k >> 2) - 1) & 1));
      if (!ok) break;
      ptx::tc_fence_after();
      const uint64_t da = da0 + static_cast<uint64_t>(s) * (kPrepTile >> 4);
      const uint32_t acc = tmem + buf * 128;
      if (ptx::elect_one()) {
        ptx::mma_ss_i<0>(acc, da, db, kIdesc);
#pragma unroll
        for (int kk = 1; kk < kFp8D / 16; ++kk) {
          const uint64_t o = (kk >> 2) * (kPrepChunk >> 4) + (kk & 3) * 2;
          ptx::mma_ss_i<1>(acc, da + o, db + o, kIdesc);
        }
        ptx::tc_commit(ba(bars.acc_full[buf]));
        ptx::tc_commit(ba(bars.empty[s]));
      }
      __syncwarp();
    }
    // every product issued completes before tensor memory is freed
    if (ptx::elect_one()) ptx::tc_commit(ba(bars.drain));
    __syncwarp();
    w.drain(ba(bars.drain), 0);
    __syncwarp();
  } else {
    // ================================================================ epilogue
    // After a failed wait the warps keep walking the items (every wait then returns at
    // once), so that the four warps always meet the same named barriers.
    const int quarter = warp & 3;  // tensor-memory lane quarter of this warp
    const int grp = (warp - 2) >> 2, ew = (warp - 2) & 3;
    const int c = quarter * 32 + lane;  // row (Q, K) or column (V) of this thread
    bool ok = true;
    for (int it = blockIdx.x + grp * gridDim.x, k = grp; it < n_items; it += 2 * gridDim.x, k += 2) {
      const int which = it / per, rem = it - which * per;
      const int bh = rem / p.n_tiles, tile = rem - bh * p.n_tiles;
      const int s = k % kPrepStages;
      float x[128];
      float amax = 0.f;
      if (which < 2) {
        const int buf = k & 3;
        ok = ok && __all_sync(0xffffffffu, w.wait(ba(bars.acc_full[buf]), (k >> 2) & 1));
        if (ok) {
          ptx::tc_fence_after();
          uint32_t raw[128];
          ptx::tmem_ld128(tmem + buf * 128 + (static_cast<uint32_t>(quarter * 32) << 16), raw);
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            x[i] = __uint_as_float(raw[i]);
            amax = fmaxf(amax, fabsf(x[i]));
          }
          ptx::tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ba(bars.acc_empty[buf]));
      } else {
        ok = ok && __all_sync(0xffffffffu, w.wait(ba(bars.full[s]), (k / kPrepStages) & 1));
        if (ok) {
          // column c: chunk c / 64, 16-byte granule (c mod 64) / 8 of each 128-byte row,
          // swizzled by row mod 8
          const uint32_t col_base = sbase + kPrepOffRing + s * kPrepTile + (c >> 6) * kPrepChunk + (c & 7) * 2;
          const int gran = (c & 63) >> 3;
#pragma unroll
          for (int r = 0; r < 128; ++r) {
            uint16_t bits;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(bits) : "r"(col_base + r * 128 + ((gran ^ (r & 7)) << 4)));
            x[r] = __uint_as_float(static_cast<uint32_t>(bits) << 16);
            amax = fmaxf(amax, fabsf(x[r]));
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const int par = (k >> 1) & 1;  // also the group's code buffer for this item
      const bool leader = ew == 0 && lane == 0;
      if (lane == 0) warp_max[grp][par][ew] = amax;
      if (leader) ptx::bulk_wait_read<1>();  // the store of two items ago has left this buffer
      ptx::named_barrier(1 + grp, 128);
      if (which == 2 && leader) ptx::mbar_arrive(ba(bars.empty[s]));  // every column has been read
      // A warp whose wait failed skips the work but not the barriers, so that the four warps
      // of the group always meet the same two barriers per item.
      if (ok) {
        amax = fmaxf(fmaxf(warp_max[grp][par][0], warp_max[grp][par][1]),
                     fmaxf(warp_max[grp][par][2], warp_max[grp][par][3]));
        const float inv = amax > 0.f ? 448.f / amax : 1.f;
        float* scales = which == 0 ? p.scales[0] : (which == 1 ? p.scales[1] : p.scales[2]);
        if (c == 0) {
          const float sc = which < 2 ? amax * 0.08838834764831845f : amax;  // Q, K: max|X R^T| / sqrt(128)
          scales[static_cast<size_t>(bh) * p.n_tiles + tile] = amax > 0.f ? sc / 448.f : 1.f;
        }
        // Q, K: row c of the tile (rows past N hold zero codes); V: row c of the transposed
        // tile.  Granule g of row c sits at position g ^ (c mod 8) (the tensor map's 128-byte
        // swizzle).
        const uint32_t row_addr = sbase + kPrepOffStage + (grp * 2 + par) * (128 * 128) + c * 128;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint32_t wd[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            wd[i] = ptx::pack_e4m3x4(x[16 * g + 4 * i] * inv, x[16 * g + 4 * i + 1] * inv,
                                     x[16 * g + 4 * i + 2] * inv, x[16 * g + 4 * i + 3] * inv);
          ptx::st_shared_v4(row_addr + ((g ^ (c & 7)) << 4), wd[0], wd[1], wd[2], wd[3]);
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::named_barrier(1 + grp, 128);
      if (ok && leader) {
        const uint32_t src = sbase + kPrepOffStage + (grp * 2 + par) * (128 * 128);
        if (which == 0) ptx::tma_store_3d(&tm_q8, src, 0, tile * 128, bh);
        else if (which == 1) ptx::tma_store_3d(&tm_k8, src, 0, tile * 128, bh);
        else ptx::tma_store_3d(&tm_vt8, src, tile * 128, 0, bh);
        ptx::bulk_commit();
      }
    }
    if (ew == 0 && lane == 0) ptx::bulk_wait_all();  // the stores have completed before the CTA exits
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kPrepTmemCols);
  }
}

// ==================================================================== attention
struct Fp8Cfg {
  static constexpr int kTileBytes = 128 * 128;  // 128 rows x 128 E4M3
  static constexpr int kSlots = 10;             // K_0, Vt_0, K_1, Vt_1, ...
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffTab = kOffRing + kSlots * kTileBytes;  // per K/V tile: s_k, log2 gain, 1/gain
  static constexpr int kTabBytes = 3 * kFp8MaxKvTiles * 4;
  static constexpr int kOffBar = kOffTab + kTabBytes;
  static constexpr int kBarQ = 0;
  static constexpr int kBarFull = 1;
  static constexpr int kBarEmpty = kBarFull + kSlots;
  static constexpr int kBarSFull = kBarEmpty + kSlots;
  static constexpr int kBarOFinal = kBarSFull + 2;
  static constexpr int kBarDrain = kBarOFinal + 2;
  static constexpr int kBarTab = kBarDrain + 1;
  static constexpr int kNumBars = kBarTab + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag, s_v max
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S_t at t * 128; P8_t over its first 32 columns
  static constexpr uint32_t kColO = 256;  // O_t at 256 + t * 128
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Fp8Params {
  const float* scale_q;  // [BH, n_tiles]
  const float* scale_k;
  const float* scale_v;
  float* lse;            // [BH, N]
  int BH, N, n_tiles, n_cta_q;
  float scale;
  float scale_log2;      // scale * log2(e)
  int causal;
  int withhold;          // test hook: the producer never loads Vt_0
  unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(kFp8Threads, 1)
    fa_fp8_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                      const Fp8Params p) {
  using C = Fp8Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  float* sv_max_slot = reinterpret_cast<float*>(smem + C::kOffMisc + 8);
  float* tab_sk = reinterpret_cast<float*>(smem + C::kOffTab);
  float* tab_lg = tab_sk + kFp8MaxKvTiles;  // log2(64 s_v,j / s_v,max)
  float* tab_ig = tab_lg + kFp8MaxKvTiles;  // s_v,max / (64 s_v,j)
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int bid = blockIdx.x, bh, cta_q;
  if (p.causal) {  // longest first
    cta_q = p.n_cta_q - 1 - bid / p.BH;
    bh = bid % p.BH;
  } else {
    bh = bid / p.n_cta_q;
    cta_q = bid % p.n_cta_q;
  }
  const int qt0 = 2 * cta_q, qt1 = qt0 + 1;
  const bool has1 = qt1 < p.n_tiles;
  const int n0 = p.causal ? qt0 + 1 : p.n_tiles;
  const int n1 = has1 ? (p.causal ? qt1 + 1 : p.n_tiles) : 0;
  const int nmax = n0 > n1 ? n0 : n1;

  if (warp == 8 && lane == 0) {
    ptx::mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      ptx::mbar_init(bar(C::kBarFull + s), 1);
      ptx::mbar_init(bar(C::kBarEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar(C::kBarSFull + t), 1);
      ptx::mbar_init(bar(C::kBarOFinal + t), 1);
    }
    ptx::mbar_init(bar(C::kBarDrain), 1);
    ptx::mbar_init(bar(C::kBarTab), 1);
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

  if (warp >= 8) ptx::regs_decrease<kFp8OtherRegs>();
  if (warp == 8) {
    // ================================================================ TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_vt);
      ptx::prefetch_tensormap(&tm_o);
      ptx::mbar_arrive_expect_tx(bar(C::kBarQ), (has1 ? 2 : 1) * C::kTileBytes);
      ptx::tma_load_3d(sbase + C::kOffQ, &tm_q, bar(C::kBarQ), 0, qt0 * 128, bh);
      if (has1) ptx::tma_load_3d(sbase + C::kOffQ + C::kTileBytes, &tm_q, bar(C::kBarQ), 0, qt1 * 128, bh);
    }
    // per-tile table of the K and V scales (plain loads; the softmax waits for kBarTab)
    const float* sk = p.scale_k + static_cast<size_t>(bh) * p.n_tiles;
    const float* sv = p.scale_v + static_cast<size_t>(bh) * p.n_tiles;
    float vmax = 0.f;
    for (int j = lane; j < nmax; j += 32) vmax = fmaxf(vmax, sv[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    for (int j = lane; j < nmax; j += 32) {
      tab_sk[j] = sk[j];
      const float ratio = fmaxf(sv[j] / vmax, 0x1p-60f);
      tab_lg[j] = kFp8PGainLog2 + log2f(ratio);
      tab_ig[j] = 1.f / (64.f * ratio);
    }
    if (lane == 0) *sv_max_slot = vmax;
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(C::kBarTab));
    if (lane == 0) {
      const int n_ring = 2 * nmax;
      int issued = 0;
      bool ok = true;
      for (int u = 0; u < n_ring; ++u) {
        const int slot = u % C::kSlots, use = u / C::kSlots;
        if (use > 0 && !w.wait(bar(C::kBarEmpty + slot), (use - 1) & 1)) { ok = false; break; }
        issued = u + 1;
        if (p.withhold && u == 1) continue;  // test hook: Vt_0 is never loaded
        ptx::mbar_arrive_expect_tx(bar(C::kBarFull + slot), C::kTileBytes);
        const uint32_t dst = sbase + C::kOffRing + slot * C::kTileBytes;
        if (u & 1) ptx::tma_load_3d(dst, &tm_vt, bar(C::kBarFull + slot), (u >> 1) * 128, 0, bh);  // Vt_j: keys x d
        else ptx::tma_load_3d(dst, &tm_k, bar(C::kBarFull + slot), 0, (u >> 1) * 128, bh);        // K_j
      }
      if (!ok) {
        w.drain(bar(C::kBarQ), 0);
        for (int u = issued - C::kSlots > 0 ? issued - C::kSlots : 0; u < issued; ++u)
          if (!(p.withhold && u == 1)) w.drain(bar(C::kBarFull + u % C::kSlots), (u / C::kSlots) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================================================================ MMA issuer
    // S_t = Q_t K_j^T and O_t += P8_t Vt_j^T, all operands K-major E4M3 (32 per step:
    // +32 bytes inside one 128-byte swizzle atom); P8_t from tensor memory (8 columns per
    // 32 keys).
    constexpr uint32_t kIdesc = ptx::idesc_e4m3_f32(128, 128);
    constexpr uint64_t kSlotStep = C::kTileBytes >> 4;
    const uint64_t desc_q0 = ptx::smem_desc_sw128(sbase + C::kOffQ, 16, 1024);
    const uint64_t desc_q1 = desc_q0 + kSlotStep;
    const uint64_t desc_ring = ptx::smem_desc_sw128(sbase + C::kOffRing, 16, 1024);
    bool ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarQ), 0));
    ptx::tc_fence_after();
    for (int j = 0; ok && j <= nmax; ++j) {
      const int uk = 2 * j, uv = 2 * j - 1;
      if (j >= 1) ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarFull + uv % C::kSlots), (uv / C::kSlots) & 1));
      if (!ok) break;
      bool k_ready = false;
      const uint64_t dk = desc_ring + static_cast<uint64_t>(uk % C::kSlots) * kSlotStep;
      const uint64_t dv = desc_ring + static_cast<uint64_t>((uv + C::kSlots) % C::kSlots) * kSlotStep;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int nt = t ? n1 : n0;
        if (j >= 1 && j - 1 < nt) {
          // P8_t(j-1) handed over through a hardware named barrier: tile t's four softmax
          // warps arrive, this warp waits (no timeout; the softmax warps arrive once per K/V
          // step whatever happens, and never for step j before S_t(j) is complete)
          ptx::named_barrier(4 + t, 160);
          ptx::tc_fence_after();
          const uint32_t t_o = tmem + C::kColO + t * kFp8D;
          const uint32_t t_p = tmem + C::kColS + t * 128;
          if (ptx::elect_one()) {
            if (j > 1) ptx::mma_ts_f8_i<1>(t_o, t_p, dv, kIdesc);
            else ptx::mma_ts_f8_i<0>(t_o, t_p, dv, kIdesc);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk) ptx::mma_ts_f8_i<1>(t_o, t_p + kk * 8, dv + kk * 2, kIdesc);
            if (j - 1 == nt - 1) ptx::tc_commit(bar(C::kBarOFinal + t));
          }
          __syncwarp();
        }
        if (j < nt) {
          if (!k_ready) {
            ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarFull + uk % C::kSlots), (uk / C::kSlots) & 1));
            if (!ok) break;
            ptx::tc_fence_after();
            k_ready = true;
          }
          const uint32_t t_s = tmem + C::kColS + t * 128;
          const uint64_t dq = t ? desc_q1 : desc_q0;
          if (ptx::elect_one()) {
            ptx::mma_ss_f8_i<0>(t_s, dq, dk, kIdesc);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk) ptx::mma_ss_f8_i<1>(t_s, dq + kk * 2, dk + kk * 2, kIdesc);
            ptx::tc_commit(bar(C::kBarSFull + t));
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (ptx::elect_one()) {
        if (j >= 1) ptx::tc_commit(bar(C::kBarEmpty + uv % C::kSlots));
        if (j < nmax) ptx::tc_commit(bar(C::kBarEmpty + uk % C::kSlots));
      }
      __syncwarp();
    }
    if (ptx::elect_one()) ptx::tc_commit(bar(C::kBarDrain));
    __syncwarp();
    w.drain(bar(C::kBarDrain), 0);
    __syncwarp();
  } else if (warp < 8) {
    // ================================================================ softmax warpgroups
    ptx::regs_increase<kFp8SoftmaxRegs>();
    const int t = warp >> 2, quarter = warp & 3;
    const int nt = t ? n1 : n0;
    const int qt = t ? qt1 : qt0;
    const int row = quarter * 32 + lane;
    const int qpos = qt * 128 + row;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS + t * 128;
    const uint32_t t_o = tmem + lane_off + C::kColO + t * kFp8D;
    const bool tile_exists = t == 0 || has1;
    const float sq = tile_exists ? p.scale_q[static_cast<size_t>(bh) * p.n_tiles + qt] : 1.f;
    const float c2 = p.scale_log2;
    float m_run = -INFINITY;  // running max of the true scores q'.k'
    float l_run = 0.f;        // running sum of 2^((s - m_run) * c2)
    // One arrive at the P hand-off barrier per K/V step, whatever happens; after a failed
    // wait the remaining steps only arrive (the loop after this one), each once S_t of its
    // step is complete (a wait that ignores the abort flag and ends at the deadline), so that
    // no arrival runs ahead into a later phase of the named barrier.
    bool ok = nt > 0 && __all_sync(0xffffffffu, w.wait(bar(C::kBarTab), 0));
    int j = 0;
    for (; ok && j < nt; ++j) {
      ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarSFull + t), j & 1));
      if (!ok) break;
      ptx::tc_fence_after();
      float s[128];  // raw E4M3 products; the true score is s * f
      {
        uint32_t r[128];
        ptx::tmem_ld128(t_s, r);
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(r[i]);
      }
      const float f = sq * tab_sk[j];
      const int col0 = j * 128;
      int lim = p.N - col0;
      if (p.causal && qpos - col0 + 1 < lim) lim = qpos - col0 + 1;
      if (lim < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < 124; c += 8) {
        mx0 = ptx::fmax3(mx0, s[c], s[c + 1]);
        mx1 = ptx::fmax3(mx1, s[c + 2], s[c + 3]);
        mx2 = ptx::fmax3(mx2, s[c + 4], s[c + 5]);
        mx3 = ptx::fmax3(mx3, s[c + 6], s[c + 7]);
      }
      mx0 = ptx::fmax3(mx0, s[124], s[125]);
      mx1 = ptx::fmax3(mx1, s[126], s[127]);
      const float tile_max = fmaxf(ptx::fmax3(mx0, mx1, mx2), mx3) * f;  // f > 0
      const float m_new = fmaxf(m_run, tile_max);
      const bool rescale = (m_new - m_run) * c2 > kFp8RescaleLog2Threshold;
      const float m_ref = rescale ? m_new : m_run;
      const float r_fac = rescale ? ptx::ex2_approx((m_run - m_new) * c2) : 1.f;
      // P8 = e4m3(2^(s f c2 - m_ref c2 + lg_j)) with lg_j = log2(64 s_v,j / s_v,max); the
      // sum for l is taken over the unrounded terms, each times 1 / (64 s_v,j / s_v,max)
      const float neg = (m_ref == -INFINITY ? 0.f : -m_ref * c2) + tab_lg[j];
      const float2 cfv = make_float2(c2 * f, c2 * f), negv = make_float2(neg, neg);
      __syncwarp();
      float2 se[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) se[i] = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 xa = __ffma2_rn(make_float2(s[4 * i], s[4 * i + 1]), cfv, negv);
        const float2 xb = __ffma2_rn(make_float2(s[4 * i + 2], s[4 * i + 3]), cfv, negv);
        const float e0 = ptx::ex2_approx(xa.x), e1 = ptx::ex2_approx(xa.y);
        const float e2 = ptx::ex2_approx(xb.x), e3 = ptx::ex2_approx(xb.y);
        pk[i] = ptx::pack_e4m3x4(e0, e1, e2, e3);
        se[i & 3] = __fadd2_rn(se[i & 3], __fadd2_rn(make_float2(e0, e1), make_float2(e2, e3)));
      }
      ptx::tmem_st32(t_s, pk);  // P8_t over columns [0, 32) of S_t
      const float2 se01 = __fadd2_rn(se[0], se[1]), se23 = __fadd2_rn(se[2], se[3]);
      l_run = l_run * r_fac + ((se01.x + se01.y) + (se23.x + se23.y)) * tab_ig[j];
      m_run = m_ref;
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int cc = 0; cc < kFp8D / 32; ++cc) {
          uint32_t r[32];
          ptx::tmem_ld32(t_o + cc * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * r_fac);
          ptx::tmem_st32(t_o + cc * 32, r);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      ptx::named_barrier_arrive(4 + t, 160);  // P8_t(j) handed over to the MMA warp
    }
    for (; j < nt && w.drain(bar(C::kBarSFull + t), j & 1); ++j) ptx::named_barrier_arrive(4 + t, 160);
    // ---- epilogue: O = O~ s_v,max / (64 l) -> bf16 -> shared (Q_t's buffer and the next
    // 16 KB) -> TMA store; LSE = m scale + ln l
    const size_t grow = static_cast<size_t>(bh) * p.N + qpos;
    const bool row_valid = qpos < p.N;
    const uint32_t so = sbase + C::kOffQ + t * 2 * C::kTileBytes;  // 32 KB bf16 staging per tile
    if (ok) ok = __all_sync(0xffffffffu, w.wait(bar(C::kBarOFinal + t), 0));
    const bool have = l_run > 0.f;
    const float inv_l = have ? *sv_max_slot / (64.f * l_run) : 0.f;
    const float lse_row = have ? m_run * p.scale + logf(l_run) : -INFINITY;
    // the staging area of tile 0 is Q_0 and Q_1's buffers: wait until both tiles' MMAs are done
    ptx::named_barrier(1, 256);
    if (ok && tile_exists) {
      ptx::tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < kFp8D / 32; ++cc) {
        uint32_t r[32];
        ptx::tmem_ld32(t_o + cc * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
        const uint32_t chunk_base = so + (cc >> 1) * (128 * 128) + row * 128;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int gran = (cc & 1) * 4 + g;
          ptx::st_shared_v4(chunk_base + ((gran ^ (row & 7)) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2],
                            pk[4 * g + 3]);
        }
      }
      if (row_valid) p.lse[grow] = lse_row;
      ptx::fence_proxy_async_smem();
    }
    ptx::named_barrier(2 + t, 128);
    if (ok && tile_exists && row == 0) {
      for (int c = 0; c < 2; ++c) ptx::tma_store_3d(&tm_o, so + c * (128 * 128), c * 64, qt * 128, bh);
      ptx::bulk_commit();
      ptx::bulk_wait_all();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ==================================================================== host side
namespace {

std::mutex g_fp8_dev_mutex;
int g_fp8_dev_state[kMaxDevices];
int g_fp8_sms[kMaxDevices];  // SM count per device, for the persistent preparation grid

int prepare_device_fp8() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_fp8_dev_mutex);
  if (g_fp8_dev_state[dev] == 1) return FA_OK;
  if (g_fp8_dev_state[dev] == -1) return FA_ERR_ARCH;
  const int arch = check_arch(dev);
  if (arch != FA_OK) {
    if (arch == FA_ERR_ARCH) g_fp8_dev_state[dev] = -1;
    return arch;
  }
  if (cudaFuncSetAttribute(fa_fp8_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Cfg::kSmemBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(fa_fp8_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmemBytes) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&g_fp8_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      g_fp8_sms[dev] < 1)
    return FA_ERR_CUDA;
  g_fp8_dev_state[dev] = 1;
  return FA_OK;
}

// Workspace: q8 [BH, N_pad, 128], k8 [BH, N_pad, 128], vt8 [BH, 128, N_pad] (E4M3 codes), then
// the fp32 scales of Q', K' and V [BH, N_pad / 128] each; every section 256-byte aligned.
struct Fp8Layout {
  size_t q8, k8, vt8, sq, sk, sv, total;
};

bool fp8_layout(long long BH, long long N, Fp8Layout* L) {
  const long long n_pad = (N + 127) / 128 * 128;
  const size_t codes = align256(static_cast<size_t>(BH * n_pad * kFp8D));
  const size_t sc = align256(static_cast<size_t>(BH * (n_pad / 128)) * 4);
  L->q8 = 0;
  L->k8 = codes;
  L->vt8 = 2 * codes;
  L->sq = 3 * codes;
  L->sk = L->sq + sc;
  L->sv = L->sk + sc;
  L->total = L->sv + sc;
  return true;
}

struct Fp8Problem {
  const void* q;
  const void* k;
  const void* v;
  const int8_t* signs;
  void* o;
  float* lse;
  int B, H, N, d;
  float scale;
  int causal;
  void* workspace;
  size_t workspace_bytes;
};

int validate_fp8(const Fp8Problem& pr, Fp8Layout* L) {
  if (!pr.q || !pr.k || !pr.v || !pr.signs || !pr.o || !pr.lse || !pr.workspace) return FA_ERR_ARG;
  if (pr.B < 1 || pr.H < 1 || pr.N < 1 || pr.d != kFp8D) return FA_ERR_ARG;
  if (!(pr.scale > 0.f) || !std::isfinite(pr.scale)) return FA_ERR_ARG;
  const long long BH = static_cast<long long>(pr.B) * pr.H;
  const long long n_tiles = (pr.N + 127LL) / 128;
  if (n_tiles > kFp8MaxKvTiles || BH * n_tiles * 128 * kFp8D > 2147483647LL || BH * n_tiles > 2147483647LL)
    return FA_ERR_ARG;
  fp8_layout(BH, pr.N, L);
  if (pr.workspace_bytes < L->total || (reinterpret_cast<uintptr_t>(pr.workspace) & 255u)) return FA_ERR_ARG;
  for (const void* ptr : {pr.q, pr.k, pr.v, static_cast<const void*>(pr.signs), static_cast<const void*>(pr.o),
                          static_cast<const void*>(pr.lse)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_ARG;
  const size_t tb = static_cast<size_t>(BH) * pr.N * kFp8D * 2, lb = static_cast<size_t>(BH) * pr.N * 4;
  const struct { const void* p; size_t n; } in[4] = {{pr.q, tb}, {pr.k, tb}, {pr.v, tb}, {pr.signs, kFp8D}};
  for (const auto& x : in) {
    if (overlaps(pr.o, tb, x.p, x.n) || overlaps(pr.lse, lb, x.p, x.n) || overlaps(pr.workspace, L->total, x.p, x.n))
      return FA_ERR_ARG;
  }
  if (overlaps(pr.o, tb, pr.lse, lb) || overlaps(pr.workspace, L->total, pr.o, tb) ||
      overlaps(pr.workspace, L->total, pr.lse, lb))
    return FA_ERR_ARG;
  for (const void* ptr : {pr.q, pr.k, pr.v, static_cast<const void*>(pr.signs), static_cast<const void*>(pr.o),
                          static_cast<const void*>(pr.lse), static_cast<const void*>(pr.workspace)})
    if (!is_device_pointer(ptr)) return FA_ERR_ARG;
  return FA_OK;
}

// The two kernels of a validated problem (the workspace laid out for its B*H heads).
int launch_fp8(const Fp8Problem& pr, int withhold, unsigned long long timeout_ns, cudaStream_t stream) {
  Fp8Layout L{};
  const int BH = pr.B * pr.H;
  fp8_layout(BH, pr.N, &L);
  const int n_tiles = (pr.N + 127) / 128, n_pad = n_tiles * 128;
  uint8_t* ws = static_cast<uint8_t*>(pr.workspace);
  QuantParams qp{};
  qp.scales[0] = reinterpret_cast<float*>(ws + L.sq);
  qp.scales[1] = reinterpret_cast<float*>(ws + L.sk);
  qp.scales[2] = reinterpret_cast<float*>(ws + L.sv);
  qp.signs = pr.signs;
  qp.BH = BH;
  qp.N = pr.N;
  qp.n_tiles = n_tiles;
  qp.n_pad = n_pad;
  qp.timeout_ns = timeout_ns;
  CUtensorMap mq, mk, mvt, mo, mxq, mxk, mxv;
  if (!encode_map_u8(&mq, ws + L.q8, BH, n_pad, kFp8D) || !encode_map_u8(&mk, ws + L.k8, BH, n_pad, kFp8D) ||
      !encode_map_u8(&mvt, ws + L.vt8, BH, kFp8D, n_pad) || !encode_map(&mo, pr.o, BH, pr.N, kFp8D) ||
      !encode_map(&mxq, pr.q, BH, pr.N, kFp8D) || !encode_map(&mxk, pr.k, BH, pr.N, kFp8D) ||
      !encode_map(&mxv, pr.v, BH, pr.N, kFp8D))
    return FA_ERR_LAUNCH;
  Fp8Params p{};
  p.scale_q = qp.scales[0];
  p.scale_k = qp.scales[1];
  p.scale_v = qp.scales[2];
  p.lse = pr.lse;
  p.BH = BH;
  p.N = pr.N;
  p.n_tiles = n_tiles;
  p.n_cta_q = (n_tiles + 1) / 2;
  p.scale = pr.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(pr.scale) * 1.4426950408889634);
  p.causal = pr.causal ? 1 : 0;
  p.withhold = withhold;
  p.timeout_ns = timeout_ns;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  const long long items = 3LL * BH * n_tiles;
  const int grid = static_cast<int>(items < g_fp8_sms[dev] ? items : g_fp8_sms[dev]);
  fa_fp8_prep_kernel<<<grid, kPrepThreads, kPrepSmemBytes, stream>>>(mxq, mxk, mxv, mq, mk, mvt, qp);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  fa_fp8_fwd_kernel<<<static_cast<unsigned>(BH * p.n_cta_q), kFp8Threads, Fp8Cfg::kSmemBytes, stream>>>(mq, mk, mvt,
                                                                                                       mo, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

int run_fp8(const Fp8Problem& pr, int withhold, unsigned long long timeout_ns, cudaStream_t stream) {
  Fp8Layout L{};
  int rc = validate_fp8(pr, &L);
  if (rc != FA_OK) return rc;
  rc = prepare_device_fp8();
  if (rc != FA_OK) return rc;
  return launch_fp8(pr, withhold, timeout_ns, stream);
}

// ---- pipelined host-to-host FP8 forward (fa_fwd_fp8_host): chunks of heads, each chunk's Q,
// K, V copied in on the library's copy stream, its two kernels on one of two compute streams
// (each with its own part of the workspace), its O and LSE copied out on the second copy
// stream while later chunks load and run.
struct Fp8Host {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
};
constexpr double kFp8FlopsPerSec = 1.35e15;  // the two kernels, measured on the causal N = 8192 step

int run_fp8_host(const Fp8Host& h, const Fp8Problem& pr, int groups_per_chunk, cudaStream_t stream) {
  Fp8Layout L{};
  int rc = validate_fp8(pr, &L);
  if (rc != FA_OK) return rc;
  if (!h.q || !h.k || !h.v || !h.o || !h.lse || groups_per_chunk < 0) return FA_ERR_ARG;
  const int BH = pr.B * pr.H;
  const size_t head_bytes = static_cast<size_t>(pr.N) * kFp8D * 2, tb = BH * head_bytes;
  const size_t lb = static_cast<size_t>(BH) * pr.N * 4;
  const struct { const void* p; size_t n; } in[3] = {{h.q, tb}, {h.k, tb}, {h.v, tb}};
  for (const auto& x : in)
    if (overlaps(h.o, tb, x.p, x.n) || overlaps(h.lse, lb, x.p, x.n)) return FA_ERR_ARG;
  if (overlaps(h.o, tb, h.lse, lb)) return FA_ERR_ARG;
  for (const void* ptr : {h.q, h.k, h.v, static_cast<const void*>(h.o), static_cast<const void*>(h.lse)})
    if (!is_pinned_host(ptr)) return FA_ERR_ARG;
  rc = prepare_device_fp8();
  if (rc != FA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe[dev].mu);
  HostPipe* hp = nullptr;
  rc = host_pipe(dev, &hp);
  if (rc != FA_OK) return rc;
  int sizes[kMaxChunks];
  const double bytes = 4.0 * tb + lb;  // q, k, v in; o, lse out
  const double flops = 4.0 * static_cast<double>(BH) * pr.N * pr.N * kFp8D * (pr.causal ? 0.5 : 1.0);
  const int n_chunks = chunk_sizes(BH, groups_per_chunk, bytes, flops / kFp8FlopsPerSec, sizes);
  // a part of the workspace per compute stream, laid out for the largest chunk; one stream
  // when two parts do not fit
  int largest = 0;
  for (int c = 0; c < n_chunks; ++c) largest = std::max(largest, sizes[c]);
  Fp8Layout Lc{};
  fp8_layout(largest, pr.N, &Lc);
  const size_t part = align256(Lc.total);
  const int n_streams = 2 * part <= pr.workspace_bytes ? kComputeStreams : 1;
  auto at = [](const void* base, size_t off) { return static_cast<const uint8_t*>(base) + off; };
  auto at_mut = [](void* base, size_t off) { return static_cast<uint8_t*>(base) + off; };
  if (cudaEventRecord(hp->start, stream) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int i = 0; i < kComputeStreams; ++i)
    if (cudaStreamWaitEvent(hp->comp[i], hp->start, 0) != cudaSuccess) return FA_ERR_CUDA;
  for (int c = 0, h0 = 0; c < n_chunks; h0 += sizes[c], ++c) {
    const int nh = sizes[c];
    const size_t off = h0 * head_bytes, len = nh * head_bytes;
    const size_t l_off = static_cast<size_t>(h0) * pr.N * 4, l_len = static_cast<size_t>(nh) * pr.N * 4;
    if (cudaMemcpyAsync(at_mut(const_cast<void*>(pr.q), off), at(h.q, off), len, cudaMemcpyHostToDevice, hp->in) !=
            cudaSuccess ||
        cudaMemcpyAsync(at_mut(const_cast<void*>(pr.k), off), at(h.k, off), len, cudaMemcpyHostToDevice, hp->in) !=
            cudaSuccess ||
        cudaMemcpyAsync(at_mut(const_cast<void*>(pr.v), off), at(h.v, off), len, cudaMemcpyHostToDevice, hp->in) !=
            cudaSuccess ||
        cudaEventRecord(hp->loaded[c], hp->in) != cudaSuccess)
      return FA_ERR_CUDA;
    const int si = c % n_streams;
    cudaStream_t cs = hp->comp[si];
    if (cudaStreamWaitEvent(cs, hp->loaded[c], 0) != cudaSuccess) return FA_ERR_CUDA;
    Fp8Problem sub = pr;
    sub.q = at(pr.q, off);
    sub.k = at(pr.k, off);
    sub.v = at(pr.v, off);
    sub.o = at_mut(pr.o, off);
    sub.lse = reinterpret_cast<float*>(at_mut(pr.lse, l_off));
    sub.B = 1;
    sub.H = nh;
    sub.workspace = at_mut(pr.workspace, si * part);
    sub.workspace_bytes = part;
    rc = launch_fp8(sub, 0, kDefaultTimeoutNs, cs);
    if (rc != FA_OK) return rc;
    if (cudaEventRecord(hp->computed[c], cs) != cudaSuccess || cudaStreamWaitEvent(hp->out, hp->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.o, off), at(pr.o, off), len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.lse, l_off), at(pr.lse, l_off), l_len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  if (cudaEventRecord(hp->done, hp->out) != cudaSuccess || cudaStreamWaitEvent(stream, hp->done, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

int fp8_status_word(int clear) {
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<int>(word & 0x7fffffffu);
}

}  // namespace fa

extern "C" {

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d != fa::kFp8D) return 0;
  fa::Fp8Layout L{};
  fa::fp8_layout(static_cast<long long>(B) * H, N, &L);
  return L.total;
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, const signed char* signs, void* o, float* lse,
               int B, int H, int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
  const fa::Fp8Problem pr{q, k, v, signs, o, lse, B, H, N, d, scale, causal, workspace, workspace_bytes};
  return fa::run_fp8(pr, 0, fa::kDefaultTimeoutNs, stream);
}

int fa_fwd_fp8_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                    void* q, void* k, void* v, const signed char* signs, void* o, float* lse, int B, int H, int N,
                    int d, float scale, int causal, void* workspace, size_t workspace_bytes, int groups_per_chunk,
                    cudaStream_t stream) {
  const fa::Fp8Problem pr{q, k, v, signs, o, lse, B, H, N, d, scale, causal, workspace, workspace_bytes};
  return fa::run_fp8_host(fa::Fp8Host{q_host, k_host, v_host, o_host, lse_host}, pr, groups_per_chunk, stream);
}

int fa_fwd_fp8_withheld_tile(const void* q, const void* k, const void* v, const signed char* signs, void* o,
                             float* lse, int B, int H, int N, int d, float scale, int causal, void* workspace,
                             size_t workspace_bytes, double wait_timeout_ms, cudaStream_t stream) {
  if (!(wait_timeout_ms >= 1.0 && wait_timeout_ms <= 10000.0)) return FA_ERR_ARG;
  const fa::Fp8Problem pr{q, k, v, signs, o, lse, B, H, N, d, scale, causal, workspace, workspace_bytes};
  return fa::run_fp8(pr, 1, static_cast<unsigned long long>(wait_timeout_ms * 1e6), stream);
}

}  // extern "C"
