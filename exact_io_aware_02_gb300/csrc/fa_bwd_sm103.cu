// fa_bwd_sm103.cu -- exact attention backward with recomputation (dQ, dK, dV), GB300, sm_103a.
//
// The forward keeps only O and the per-row LSE; the backward rebuilds S and P on chip
// from them (the recompute scheme of §6 of the zzszmyf.github.io notes "FlashAttention
// 原理是什么？为什么又省显存又快" and of the aiqz.cc article's 工程实现细节 section):
//     P = exp(scale*Q K^T - LSE),   D = rowsum(dO * O),
//     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),
//     dQ = scale * dS K,   dK = scale * dS^T Q.
//
// Three kernels, all on one stream:
//   fa_bwd_prep_kernel  -- D = rowsum(dO * O) (memory-bound, 16-byte loads, a row per D/8
//                          lanes);
//   fa_bwd_dkdv_kernel  -- one CTA per 128-key tile: loops over the query tiles that see
//                          it, recomputes S^T = K Q^T and dP^T = V dO^T, and accumulates
//                          dV += P^T dO and dK += dS^T Q in tensor memory;
//   fa_bwd_dq_kernel    -- one CTA per 128-query tile: loops over its key tiles,
//                          recomputes S = Q K^T and dP = dO V^T, accumulates dQ += dS K.
//                          It reads nothing the dK/dV kernel writes and is launched as its
//                          programmatic dependent, so it fills the SMs that kernel's last wave
//                          leaves idle; each of its CTAs waits for the dK/dV grid before exiting.
// Splitting dQ from dK/dV costs two extra products per tile pair (7 instead of 5) but
// needs no atomics and keeps every accumulator in tensor memory.
//
// Both main kernels: warps 0-7 compute -- warp w reads TMEM lane quarter w % 4 (one row
// per thread) and column half w / 4, so two warps share each SM sub-partition; warp 8
// is the TMA producer; warp 9 allocates tensor memory and issues the MMAs (converged
// warp, elect.sync).  The bf16 P and dS each warp produces are packed into the first
// half of the fp32 columns that warp itself has read, so no warp overwrites columns
// another warp still has to read; the MMAs that consume them address the two packed
// halves separately.  Every mbarrier wait is bounded, as in the forward.
#include "fa_common.cuh"

namespace fa {

constexpr int kBwdThreads = 320;
constexpr int kBwdComputeWarps = 8;
// The compute warps hand P^T and dS^T (dK/dV kernel) and dS (dQ kernel) to the MMA warp through
// hardware named barriers: the compute warps arrive (bar.arrive), the MMA warp waits
// (bar.sync), which wakes far sooner than an mbarrier wait.  The epilogue's barrier among the
// compute warps is ID 1.  A bar.sync has no timeout, so the compute warps arrive once per step
// whatever happens, and never for step u before the input of step u (an S or dP tile, issued
// after the MMA warp's wait for step u-1) is complete; after a failed wait of their own they
// wait for that input with a wait that ignores the abort flag and ends at the deadline.
constexpr uint32_t kNbP = 2, kNbDS = 3;
constexpr uint32_t kHandOffThreads = 32 * (kBwdComputeWarps + 1);

// ---------------------------------------------------------------- D = rowsum(dO * O)
// Memory-bound: each lane reads 16-byte pieces (8 elements) of a row of O and of dO, a row
// spans D/8 lanes, and every lane has kPrepLoads pieces of each tensor in flight.  The sum is
// formed in one fixed order: sequential fused multiply-adds over runs of D/32 elements, then a
// pairwise tree over the D/32-element runs (the partner at the largest distance first), so D is
// the same bits whatever the load width.
constexpr int kPrepThreads = 256, kPrepLoads = 4;
template <int D>
__host__ __device__ constexpr int prep_rows_per_warp() { return (32 / (D / 8)) * kPrepLoads; }

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    fa_bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                       float* __restrict__ dvec, int rows) {
  constexpr int kLanesPerRow = D / 8, kRowsPerLoad = 32 / kLanesPerRow;
  constexpr int kRun = D / 32;          // elements per sequential run
  constexpr int kRuns = 8 / kRun;       // runs per 16-byte piece
  constexpr int kWordsPerRun = kRun / 2;
  const int lane = threadIdx.x & 31;
  const long long warp_id = static_cast<long long>(blockIdx.x) * (kPrepThreads / 32) + (threadIdx.x >> 5);
  const long long row0 = warp_id * prep_rows_per_warp<D>() + lane / kLanesPerRow;
  const int piece = lane % kLanesPerRow;
  uint4 a[kPrepLoads], b[kPrepLoads];
#pragma unroll
  for (int i = 0; i < kPrepLoads; ++i) {
    const long long row = row0 + i * kRowsPerLoad;
    a[i] = b[i] = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows) {
      const size_t off = static_cast<size_t>(row) * D + piece * 8;
      a[i] = __ldg(reinterpret_cast<const uint4*>(o + off));
      b[i] = __ldg(reinterpret_cast<const uint4*>(dout + off));
    }
  }
#pragma unroll
  for (int i = 0; i < kPrepLoads; ++i) {
    const uint32_t av[4] = {a[i].x, a[i].y, a[i].z, a[i].w}, bv[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
    float part[kRuns];
#pragma unroll
    for (int r = 0; r < kRuns; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int w = r * kWordsPerRun; w < (r + 1) * kWordsPerRun; ++w) {
        acc += __uint_as_float(av[w] << 16) * __uint_as_float(bv[w] << 16);
        acc += __uint_as_float(av[w] & 0xffff0000u) * __uint_as_float(bv[w] & 0xffff0000u);
      }
      part[r] = acc;
    }
    // the tree over the row's runs: first across lanes (run distances kRuns * off), then
    // within the lane
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
#pragma unroll
      for (int r = 0; r < kRuns; ++r) part[r] += __shfl_xor_sync(0xffffffffu, part[r], off);
#pragma unroll
    for (int step = kRuns / 2; step > 0; step >>= 1)
#pragma unroll
      for (int r = 0; r < step; ++r) part[r] = part[r] + part[r + step];
    const long long row = row0 + i * kRowsPerLoad;
    if (piece == 0 && row < rows) dvec[row] = part[0];
  }
}

struct BwdParams {
  const float* lse;   // [groups * R]
  const float* dvec;  // [groups * R]
  int groups;         // B * Hkv
  int R;              // query rows per group (G * N)
  int N;              // sequence length (queries and keys)
  int n_qtiles;       // ceil(R / 128)
  int n_ktiles;       // ceil(N / 128)
  float scale;
  float scale_log2;   // scale * log2(e)
  int causal;
  int withhold;      // test hook: the dK/dV producer never loads stage 0's tiles and the dQ
                     // producer never loads V_0, so those waits can only give up
  unsigned long long timeout_ns;
};

// highest sequence position of any query row in tile qt (rows straddling heads: N - 1)
__device__ __forceinline__ int bwd_tile_max_pos(const BwdParams& p, int qt) {
  const int r0 = qt * 128;
  const int r1 = min(r0 + 127, p.R - 1);
  return (r1 / p.N != r0 / p.N) ? p.N - 1 : r1 % p.N;
}

// The query tiles of a group that reach key tile kt, in order, with the sequence position of
// each tile's first row (its row mod N) carried along.  With causal masking the tiles of a head
// that end before position kt*128 are jumped over in one step (one division per head), not
// tested one by one: a loop over every tile with divisions took a key tile's CTA several
// microseconds before its first load.
struct QTileWalk {
  int qt = 0, pos0 = 0;
  // the highest position of the tile's rows (a tile straddling heads reaches N - 1)
  __device__ __forceinline__ int max_pos(const BwdParams& p) const {
    const int last = pos0 + min(128, p.R - qt * 128) - 1;
    return last >= p.N ? p.N - 1 : last;
  }
  // from the current tile to the first that reaches key tile kt: a tile that does not lies in
  // one head, below position kt*128, and the tile holding that position of the same head does
  __device__ __forceinline__ void seek(const BwdParams& p, int kt) {
    if (!p.causal) return;
    while (qt < p.n_qtiles && max_pos(p) < kt * 128) {
      const int head_row0 = qt * 128 - pos0;
      const int to = (head_row0 + kt * 128) / 128;
      pos0 += (to - qt) * 128;
      qt = to;
    }
  }
  __device__ __forceinline__ void next(const BwdParams& p, int kt) {
    ++qt;
    pos0 += 128;
    while (pos0 >= p.N) pos0 -= p.N;
    seek(p, kt);
  }
};

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kVecBytes = 2 * 128 * 4;     // -LSE*log2(e) and -D of one query tile
  // dK/dV kernel: K, V resident; a ring of stages {Q_i, dO_i, -LSE_i log2 e, -D_i}
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kStageBytes = 2 * kTileBytes + kVecBytes;
  static constexpr int kKVOffStage = 2 * kTileBytes;
  static constexpr int kKVOffBar = kKVOffStage + kStages * kStageBytes;
  // dQ kernel: Q, dO resident; a ring of K_j, V_j tiles
  static constexpr int kSlots = D == 128 ? 5 : 12;
  static constexpr int kPrefetchAhead = 4;  // producer tiles fetched into L2 ahead of their load
  static constexpr int kQOffRing = 2 * kTileBytes;
  static constexpr int kQOffBar = kQOffRing + kSlots * kTileBytes;
  static constexpr int kMaxBars = 2 + 2 * (kSlots > kStages ? kSlots : kStages) + 8;
  static constexpr int kSmemKV = kKVOffBar + kMaxBars * 8 + 16 + 1024;
  static constexpr int kSmemQ = kQOffBar + kMaxBars * 8 + 16 + 1024;
  // dK/dV kernel tensor memory: S^T, dP^T, dV, dK
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
  // dQ kernel tensor memory: two S buffers (key tiles alternate), dP, dQ
  static constexpr uint32_t kQColS = 0, kQColDP = 256, kQColDQ = 384;
  static_assert(kSmemKV <= 232448 && kSmemQ <= 232448, "shared memory budget");
};

// MMA helpers shared by both kernels -------------------------------------------------
// C[tmem, 128 x 128] = A (128 rows x D, K-major smem) * B^T (128 rows x D, K-major smem)
template <int D>
__device__ __forceinline__ void bwd_mma_nt(uint32_t c, uint64_t da, uint64_t db) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false);
  ptx::mma_ss_i<0>(c, da, db, idesc);
#pragma unroll
  for (int kk = 1; kk < D / 16; ++kk) {
    const uint64_t o = (kk >> 2) * (BwdCfg<D>::kChunkBytes >> 4) + (kk & 3) * 2;
    ptx::mma_ss_i<1>(c, da + o, db + o, idesc);
  }
}
// C[tmem, 128 x D] (+)= A * B: A is 128 x 128 bf16 in tensor memory, packed by the two
// column halves (inner index 0..63 at columns [0, 32), 64..127 at [64, 96)); B is
// 128 rows x D, N-contiguous in shared memory.
template <int D>
__device__ __forceinline__ void bwd_mma_tn(uint32_t c, uint32_t a_tmem, uint64_t db, bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, D, true);
  if (accumulate) ptx::mma_ts_i<1>(c, a_tmem, db, idesc);
  else ptx::mma_ts_i<0>(c, a_tmem, db, idesc);
#pragma unroll
  for (int kk = 1; kk < 8; ++kk)
    ptx::mma_ts_i<1>(c, a_tmem + (kk >> 2) * 64 + (kk & 3) * 8, db + kk * 128, idesc);
}

// The dK/dV kernel's first elementwise step for this thread's key row, over this warp's
// 64 query columns: P^T = exp2(S^T * scale*log2(e) - LSE*log2(e)) into pr[] (fp32) and,
// rounded to bf16 pairs, into tensor memory over the first 32 of the columns read.
// kMasked adds the per-element test (key exists, query row exists, causal order);
// tiles that need none take the kMasked = false instance.
// Start a load of 32 consecutive 32-bit TMEM columns of this warp's lanes; the registers are
// valid only after bwd_wait_ld32 on the same array (which waits for every load in flight).
__device__ __forceinline__ void bwd_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void bwd_wait_ld32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Convert columns [c0, c0 + D/2) of kN 128-row fp32 accumulators (this thread's row), each
// times its own factor, to bf16 in 128B-swizzled shared tiles (the TMA layout).  Every
// tensor-memory load is issued before the first is waited for: one round trip in all, not one
// per 32 columns.
template <int D, int kN>
__device__ __forceinline__ void bwd_accs_to_smem(const uint32_t (&t_acc)[kN], const uint32_t (&smem_tile)[kN],
                                                 const float (&mul)[kN], int row, int c0) {
  constexpr int kC = D / 64;  // 32-column chunks per accumulator in this thread's half
  uint32_t r[kN][kC][32];
#pragma unroll
  for (int n = 0; n < kN; ++n)
#pragma unroll
    for (int cc = 0; cc < kC; ++cc) bwd_ld32_nowait(t_acc[n] + c0 + 32 * cc, r[n][cc]);
#pragma unroll
  for (int n = 0; n < kN; ++n)
#pragma unroll
    for (int cc = 0; cc < kC; ++cc) {
      bwd_wait_ld32(r[n][cc]);  // the first waits for every load; the others only order the registers
      const int chunk = c0 / 32 + cc;  // 32-column chunk of the row
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = ptx::pack_bf16x2(__uint_as_float(r[n][cc][2 * i]) * mul[n], __uint_as_float(r[n][cc][2 * i + 1]) * mul[n]);
      const uint32_t base = smem_tile[n] + (chunk >> 1) * BwdCfg<D>::kChunkBytes + row * 128;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int gran = (chunk & 1) * 4 + g;
        ptx::st_shared_v4(base + ((gran ^ (row & 7)) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
      }
    }
}

template <bool kMasked>
__device__ __forceinline__ void bwd_kv_p(uint32_t t_s, const float* vec, int col0, float c2, int key,
                                         bool key_valid, int n_rows, int pos0, int N, bool causal,
                                         float (&pr)[64]) {
  // two 32-column halves: the first half's terms are computed and stored while the second lands
  uint32_t r[2][32];
  bwd_ld32_nowait(t_s, r[0]);
  bwd_wait_ld32(r[0]);
  bwd_ld32_nowait(t_s + 32, r[1]);
  const float2 c2v = make_float2(c2, c2);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c == 1) bwd_wait_ld32(r[1]);
#pragma unroll
    for (int i = 32 * c; i < 32 * c + 32; i += 4) {
      const float4 nl = *reinterpret_cast<const float4*>(vec + col0 + i);
      const float nla[4] = {nl.x, nl.y, nl.z, nl.w};
#pragma unroll
      for (int h = 0; h < 4; h += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[c][i - 32 * c + h]),
                                                __uint_as_float(r[c][i - 32 * c + h + 1])),
                                    c2v, make_float2(nla[h], nla[h + 1]));
        float e[2] = {ptx::ex2_approx(x.x), ptx::ex2_approx(x.y)};
        if constexpr (kMasked) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int col = col0 + i + h + t;
            const int qpos = (pos0 + col) % N;
            e[t] = (key_valid && col < n_rows && !(causal && qpos < key)) ? e[t] : 0.f;
          }
        }
        pr[i + h] = e[0];
        pr[i + h + 1] = e[1];
      }
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16x2(pr[32 * c + 2 * i], pr[32 * c + 2 * i + 1]);
    ptx::tmem_st16(t_s + 16 * c, pk);
  }
}

// The second step, shared by both kernels: dS = P * (dP - D) over this warp's 64 columns
// (dP read from t_dp; -D per column from neg_dcol[], or one -D for the whole row), rounded
// to bf16 pairs into 32 tensor-memory columns at t_dst (columns this warp has read).
template <bool kPerColumnD>
__device__ __forceinline__ void bwd_ds(uint32_t t_dp, uint32_t t_dst, const float (&pr)[64], const float* neg_dcol,
                                       float neg_drow) {
  // two 32-column halves: the first half's dS is computed and stored while the second lands
  uint32_t r[2][32];
  bwd_ld32_nowait(t_dp, r[0]);
  bwd_wait_ld32(r[0]);
  bwd_ld32_nowait(t_dp + 32, r[1]);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c == 1) bwd_wait_ld32(r[1]);
    float ds[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float nd[4] = {neg_drow, neg_drow, neg_drow, neg_drow};
      if constexpr (kPerColumnD) {
        const float4 d4 = *reinterpret_cast<const float4*>(neg_dcol + 32 * c + i);
        nd[0] = d4.x; nd[1] = d4.y; nd[2] = d4.z; nd[3] = d4.w;
      }
#pragma unroll
      for (int h = 0; h < 4; h += 2) {
        const float2 t = __fadd2_rn(make_float2(__uint_as_float(r[c][i + h]), __uint_as_float(r[c][i + h + 1])),
                                    make_float2(nd[h], nd[h + 1]));
        const float2 q = __fmul2_rn(make_float2(pr[32 * c + i + h], pr[32 * c + i + h + 1]), t);
        ds[i + h] = q.x;
        ds[i + h + 1] = q.y;
      }
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16x2(ds[2 * i], ds[2 * i + 1]);
    ptx::tmem_st16(t_dst + 16 * c, pk);
  }
}

// ================================================================ dK, dV
// CTA (group bh, key tile kt).  Tensor memory: S^T [0,128) with P^T packed into
// [0,32) and [64,96), dP^T [128,256) with dS^T packed the same way, dV, dK after that.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  // barriers: 0 kv_full, [1, 1+S) stage_full, [1+S, 1+2S) stage_empty, then S^T ready,
  // dP^T ready, P^T written, dS^T written, accumulators final, drain
  constexpr int S = C::kStages;
  constexpr int kBarKV = 0, kBarFull = 1, kBarEmpty = 1 + S, kBarS = 1 + 2 * S, kBarDP = kBarS + 1,
                kBarFinal = kBarDP + 1, kBarDrain = kBarFinal + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kKVOffBar + C::kMaxBars * 8);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kKVOffBar + C::kMaxBars * 8 + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kKVOffBar + 8u * i; };
  auto stage_addr = [&](int s) -> uint32_t { return sbase + C::kKVOffStage + s * C::kStageBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x % p.groups;
  const int kt = blockIdx.x / p.groups;  // causal: the first key tiles have the most work, so go first
  // the query tiles that see this key tile (causal: some position >= kt*128), counted once by
  // the producer warp and shared
  volatile int* n_q_slot = reinterpret_cast<volatile int*>(smem + C::kKVOffBar + C::kMaxBars * 8 + 8);
  // the dQ kernel, which reads nothing this grid writes, may take the SMs this grid leaves idle
  ptx::griddep_launch_dependents();

  // Producer state, carried across the set-up barrier: the walk over the query tiles and the
  // LSE and D of the next tile's rows (loaded one tile ahead, so their latency hides behind the
  // set-up and then behind each stage's wait)
  QTileWalk qw;
  float lse_next[4], d_next[4];
  auto load_vec = [&](int qt) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = qt * 128 + lane + 32 * j;
      const size_t g = static_cast<size_t>(bh) * p.R + (r < p.R ? r : 0);
      lse_next[j] = r < p.R ? __ldg(p.lse + g) : 0.f;
      d_next[j] = r < p.R ? __ldg(p.dvec + g) : 0.f;
    }
  };
  if (warp == kBwdComputeWarps) {
    qw.seek(p, kt);
    load_vec(qw.qt);
    // the count, a tile per lane at a time
    int count = 0;
    for (int qt = lane; qt < p.n_qtiles; qt += 32) count += (!p.causal || bwd_tile_max_pos(p, qt) >= kt * 128) ? 1 : 0;
    count = __reduce_add_sync(0xffffffffu, count);
    if (lane == 0) {
      ptx::mbar_init(bar(kBarKV), 1);
      for (int s = 0; s < S; ++s) {
        ptx::mbar_init(bar(kBarFull + s), 2);  // TMA bytes + the producer's LSE/D stores
        ptx::mbar_init(bar(kBarEmpty + s), 1);
      }
      ptx::mbar_init(bar(kBarS), 1);
      ptx::mbar_init(bar(kBarDP), 1);
      ptx::mbar_init(bar(kBarFinal), 1);
      ptx::mbar_init(bar(kBarDrain), 1);
      *abort_flag = 0u;
      *n_q_slot = count;
      ptx::fence_mbar_init();
      // K, V and the first query tile's Q, dO start loading before the set-up barrier
      ptx::mbar_arrive_expect_tx(bar(kBarKV), 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        ptx::tma_load_3d(sbase + c * C::kChunkBytes, &tm_k, bar(kBarKV), c * 64, kt * 128, bh);
        ptx::tma_load_3d(sbase + C::kTileBytes + c * C::kChunkBytes, &tm_v, bar(kBarKV), c * 64, kt * 128, bh);
      }
      if (count > 0 && !p.withhold) {
        ptx::mbar_arrive_expect_tx(bar(kBarFull), 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          ptx::tma_load_3d(stage_addr(0) + c * C::kChunkBytes, &tm_q, bar(kBarFull), c * 64, qw.qt * 128, bh);
          ptx::tma_load_3d(stage_addr(0) + C::kTileBytes + c * C::kChunkBytes, &tm_do, bar(kBarFull), c * 64,
                           qw.qt * 128, bh);
        }
      }
    }
  }
  if (warp == kBwdComputeWarps + 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_q = *n_q_slot;
  const Waiter w{abort_flag, p.timeout_ns};
  constexpr float kLog2e = 1.4426950408889634f;

  if (warp == kBwdComputeWarps) {
    // ------------------------------------------------ producer: stages of Q, dO, -LSE log2 e, -D
    // (K, V and stage 0's Q, dO were issued before the set-up barrier)
    int u = 0, issued = 0;
    bool ok = true;
    while (qw.qt < p.n_qtiles) {
      const int qt = qw.qt;
      const int s = u % S, use = u / S;
      if (use > 0) ok = __all_sync(0xffffffffu, w.wait(bar(kBarEmpty + s), (use - 1) & 1));
      if (!ok) break;
      const uint32_t st = stage_addr(s);
      if (lane == 0 && u > 0) {
        ptx::mbar_arrive_expect_tx(bar(kBarFull + s), 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          ptx::tma_load_3d(st + c * C::kChunkBytes, &tm_q, bar(kBarFull + s), c * 64, qt * 128, bh);
          ptx::tma_load_3d(st + C::kTileBytes + c * C::kChunkBytes, &tm_do, bar(kBarFull + s), c * 64, qt * 128, bh);
        }
      }
      // the loaded LSE and D are first used here, after the tile's loads are on their way
      asm volatile("" : "+f"(lse_next[0]), "+f"(lse_next[1]), "+f"(lse_next[2]), "+f"(lse_next[3]),
                   "+f"(d_next[0]), "+f"(d_next[1]), "+f"(d_next[2]), "+f"(d_next[3]));
      float* vec = reinterpret_cast<float*>(smem + C::kKVOffStage + s * C::kStageBytes + 2 * C::kTileBytes);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool row_exists = qt * 128 + lane + 32 * j < p.R;  // padding rows: 0
        vec[lane + 32 * j] = row_exists ? -lse_next[j] * kLog2e : 0.f;
        vec[128 + lane + 32 * j] = row_exists ? -d_next[j] : 0.f;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarFull + s));
      ++u;
      issued = u;
      qw.next(p, kt);
      if (qw.qt < p.n_qtiles) load_vec(qw.qt);
    }
    if (!ok && lane == 0) {
      w.drain(bar(kBarKV), 0);
      for (int v = issued - S > 0 ? issued - S : 0; v < issued; ++v)
        if (!(p.withhold && v == 0)) w.drain(bar(kBarFull + v % S), (v / S) & 1);
    }
    __syncwarp();
  } else if (warp == kBwdComputeWarps + 1) {
    // ------------------------------------------------ MMA issuer
    const uint64_t desc_k = ptx::smem_desc_sw128(sbase, 16, 1024);
    const uint64_t desc_v = ptx::smem_desc_sw128(sbase + C::kTileBytes, 16, 1024);
    const uint64_t desc_stage_kmaj = ptx::smem_desc_sw128(stage_addr(0), 16, 1024);
    const uint64_t desc_stage_nmaj = ptx::smem_desc_sw128(stage_addr(0), C::kChunkBytes, 1024);
    constexpr uint64_t kStageStep = C::kStageBytes >> 4, kTileStep = C::kTileBytes >> 4;
    const uint32_t t_s = tmem + C::kColS, t_dp = tmem + C::kColDP;
    const uint32_t t_dv = tmem + C::kColAcc0, t_dk = tmem + C::kColAcc1;
    // Per query tile u: S^T(u), dP^T(u) | wait P^T(u): dV(u), S^T(u+1) | wait dS^T(u):
    // dK(u), dP^T(u+1).  S^T(u+1) overwrites P^T(u) only after dV(u) read it, and dP^T(u+1)
    // overwrites dS^T(u) only after dK(u): the tensor pipe runs one CTA's MMAs in order.
    bool ok = __all_sync(0xffffffffu, w.wait(bar(kBarKV), 0));
    ptx::tc_fence_after();
    if (ok && n_q > 0) {
      ok = __all_sync(0xffffffffu, w.wait(bar(kBarFull), 0));
      if (ok) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          bwd_mma_nt<D>(t_s, desc_k, desc_stage_kmaj);                // S^T = K Q^T
          ptx::tc_commit(bar(kBarS));
          bwd_mma_nt<D>(t_dp, desc_v, desc_stage_kmaj + kTileStep);   // dP^T = V dO^T
          ptx::tc_commit(bar(kBarDP));
        }
        __syncwarp();
      }
    }
    for (int u = 0; ok && u < n_q; ++u) {
      const int s = u % S, s1 = (u + 1) % S;
      const bool more = u + 1 < n_q;
      const uint64_t st_n = desc_stage_nmaj + s * kStageStep;
      ptx::named_barrier(kNbP, kHandOffThreads);  // P^T(u) written
      ptx::tc_fence_after();
      if (ptx::elect_one()) bwd_mma_tn<D>(t_dv, t_s, st_n + kTileStep, u > 0);  // dV += P^T dO
      __syncwarp();
      if (more) {
        ok = __all_sync(0xffffffffu, w.wait(bar(kBarFull + s1), ((u + 1) / S) & 1));
        if (!ok) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          bwd_mma_nt<D>(t_s, desc_k, desc_stage_kmaj + s1 * kStageStep);
          ptx::tc_commit(bar(kBarS));
        }
        __syncwarp();
      }
      ptx::named_barrier(kNbDS, kHandOffThreads);  // dS^T(u) written
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        bwd_mma_tn<D>(t_dk, t_dp, st_n, u > 0);  // dK += dS^T Q (scaled in the epilogue)
        ptx::tc_commit(bar(kBarEmpty + s));
        if (more) {
          bwd_mma_nt<D>(t_dp, desc_v, desc_stage_kmaj + s1 * kStageStep + kTileStep);
          ptx::tc_commit(bar(kBarDP));
        } else {
          ptx::tc_commit(bar(kBarFinal));
        }
      }
      __syncwarp();
    }
    if (ptx::elect_one()) ptx::tc_commit(bar(kBarDrain));
    __syncwarp();
    w.drain(bar(kBarDrain), 0);
    __syncwarp();
  } else {
    // ------------------------------------------------ compute: thread = key row, warp = column half
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int key = kt * 128 + row;
    const bool key_valid = key < p.N;
    const bool key_tile_full = kt * 128 + 128 <= p.N;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS + half * 64, t_dp = tmem + lane_off + C::kColDP + half * 64;
    const float c2 = p.scale_log2;
    bool ok = true;
    int u = 0, np = 0;  // query tiles whose dS^T (P^T) has been handed over
    QTileWalk walk;
    for (walk.seek(p, kt); walk.qt < p.n_qtiles && ok; walk.next(p, kt)) {
      const int qt = walk.qt;
      const int s = u % S;
      // the tile needs no mask when all 128 rows exist, all keys exist and (causal) its
      // lowest position is at or after the key tile's last key
      const int r0 = qt * 128;
      const int n_rows = min(128, p.R - r0);
      const int pos0 = walk.pos0;
      const bool one_head = pos0 + 128 <= p.N;
      const bool no_mask = n_rows == 128 && key_tile_full && (!p.causal || (one_head && pos0 >= kt * 128 + 127));
      ok = __all_sync(0xffffffffu, w.wait(bar(kBarS), u & 1));
      if (!ok) break;
      ptx::tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(smem + C::kKVOffStage + s * C::kStageBytes + 2 * C::kTileBytes);
      float pr[64];
      if (no_mask)
        bwd_kv_p<false>(t_s, vec, half * 64, c2, key, key_valid, n_rows, pos0, p.N, p.causal, pr);
      else
        bwd_kv_p<true>(t_s, vec, half * 64, c2, key, key_valid, n_rows, pos0, p.N, p.causal, pr);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      ptx::named_barrier_arrive(kNbP, kHandOffThreads);  // P^T(u) handed over
      np = u + 1;
      ok = __all_sync(0xffffffffu, w.wait(bar(kBarDP), u & 1));
      if (!ok) break;
      ptx::tc_fence_after();
      bwd_ds<true>(t_dp, t_dp, pr, vec + 128 + half * 64, 0.f);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      ptx::named_barrier_arrive(kNbDS, kHandOffThreads);  // dS^T(u) handed over
      ++u;
    }
    // after a failed wait: the remaining arrivals, each once the input of its step is complete
    for (; u < n_q; ++u) {
      if (np == u) {
        if (!w.drain(bar(kBarS), u & 1)) break;
        ptx::named_barrier_arrive(kNbP, kHandOffThreads);
        ++np;
      }
      if (!w.drain(bar(kBarDP), u & 1)) break;
      ptx::named_barrier_arrive(kNbDS, kHandOffThreads);
    }
    // epilogue: dV, scale*dK -> bf16 -> shared (K and V buffers, no longer read) -> TMA
    if (ok && n_q > 0) ok = __all_sync(0xffffffffu, w.wait(bar(kBarFinal), 0));
    if (ok && n_q > 0) {
      ptx::tc_fence_after();
      const uint32_t t_acc[2] = {tmem + lane_off + C::kColAcc0, tmem + lane_off + C::kColAcc1};  // dV, dK
      const uint32_t dst[2] = {sbase + C::kTileBytes, sbase};
      const float mul[2] = {1.f, p.scale};
      bwd_accs_to_smem<D, 2>(t_acc, dst, mul, row, half * (D / 2));
      ptx::fence_proxy_async_smem();
    } else if (n_q == 0 && ok) {
      // no query sees this key tile: zero gradients (the K/V tiles may still be landing)
      ok = __all_sync(0xffffffffu, w.wait(bar(kBarKV), 0));
      if (ok) {
        const int t = threadIdx.x;  // 0..255
        for (int i = 0; i < 2 * C::kTileBytes / 16; i += 32 * kBwdComputeWarps)
          ptx::st_shared_v4(sbase + (i + t) * 16, 0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
      }
    }
    ptx::named_barrier(1, 32 * kBwdComputeWarps);
    if (ok && threadIdx.x == 0) {
      for (int c = 0; c < C::kChunks; ++c) {
        ptx::tma_store_3d(&tm_dk, sbase + c * C::kChunkBytes, c * 64, kt * 128, bh);
        ptx::tma_store_3d(&tm_dv, sbase + C::kTileBytes + c * C::kChunkBytes, c * 64, kt * 128, bh);
      }
      ptx::bulk_commit();
      ptx::bulk_wait_read<0>();  // the stores have read their staging: the CTA may exit
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdComputeWarps + 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ================================================================ dQ
// CTA (group bh, query tile qt).  Tensor memory: S of even key tiles [0,128), of odd key
// tiles [128,256); dP [256,384); dQ after that.  dS(j) is packed over the S(j) columns
// the P step has read, so S(j+1) is already resident while dS(j) is computed.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  constexpr int S = C::kSlots;
  // barriers: 0 Q/dO, [1, 1+S) ring full, [1+S, 1+2S) ring empty, then S ready (one per
  // S buffer), dP ready, dS written, dQ final, drain
  constexpr int kBarQ = 0, kBarFull = 1, kBarEmpty = 1 + S, kBarS = 1 + 2 * S, kBarDP = kBarS + 2,
                kBarFinal = kBarDP + 1, kBarDrain = kBarFinal + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kQOffBar + C::kMaxBars * 8);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kQOffBar + C::kMaxBars * 8 + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kQOffBar + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x % p.groups;
  const int qt = p.n_qtiles - 1 - blockIdx.x / p.groups;  // causal: the last query tiles have most work
  const int n_kv = p.causal ? min(p.n_ktiles, bwd_tile_max_pos(p, qt) / 128 + 1) : p.n_ktiles;
  // compute threads: the LSE and D of this thread's query row, loaded before the set-up barrier
  const int qrow = qt * 128 + (warp & 3) * 32 + lane;
  const bool row_valid = qrow < p.R;
  float lse_row = 0.f, d_row = 0.f;
  if (warp < kBwdComputeWarps && row_valid) {
    const size_t g = static_cast<size_t>(bh) * p.R + qrow;
    lse_row = __ldg(p.lse + g);
    d_row = __ldg(p.dvec + g);
  }
  // producer (warp 8, lane 0): ring tiles issued so far, carried across the set-up barrier
  int issued = 0;
  auto prefetch = [&](int u) {
    if (u < 2 * n_kv)
      for (int c = 0; c < C::kChunks; ++c)
        ptx::tma_prefetch_3d((u & 1) ? &tm_v : &tm_k, c * 64, (u >> 1) * 128, bh);
  };
  auto load_ring = [&](int u) {  // K_{u/2} (u even) or V_{u/2} (u odd) into slot u % S
    const int s = u % S;
    ptx::mbar_arrive_expect_tx(bar(kBarFull + s), C::kTileBytes);
    for (int c = 0; c < C::kChunks; ++c)
      ptx::tma_load_3d(sbase + C::kQOffRing + s * C::kTileBytes + c * C::kChunkBytes, (u & 1) ? &tm_v : &tm_k,
                       bar(kBarFull + s), c * 64, (u >> 1) * 128, bh);
  };

  if (warp == kBwdComputeWarps && lane == 0) {
    ptx::mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(bar(kBarFull + s), 1);
      ptx::mbar_init(bar(kBarEmpty + s), 1);
    }
    ptx::mbar_init(bar(kBarS), 1);
    ptx::mbar_init(bar(kBarS + 1), 1);
    ptx::mbar_init(bar(kBarDP), 1);
    ptx::mbar_init(bar(kBarFinal), 1);
    ptx::mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
    // Q, dO and the ring's first tiles (no slot to wait for yet) start loading before the
    // set-up barrier
    ptx::mbar_arrive_expect_tx(bar(kBarQ), 2 * C::kTileBytes);
    for (int c = 0; c < C::kChunks; ++c) {
      ptx::tma_load_3d(sbase + c * C::kChunkBytes, &tm_q, bar(kBarQ), c * 64, qt * 128, bh);
      ptx::tma_load_3d(sbase + C::kTileBytes + c * C::kChunkBytes, &tm_do, bar(kBarQ), c * 64, qt * 128, bh);
    }
    for (int u = 0; u < C::kPrefetchAhead; ++u) prefetch(u);
    for (int u = 0; u < S && u < 2 * n_kv; ++u) {
      prefetch(u + C::kPrefetchAhead);
      issued = u + 1;
      if (p.withhold && u == 1) continue;  // test hook: V_0 is never loaded
      load_ring(u);
    }
  }
  if (warp == kBwdComputeWarps + 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter w{abort_flag, p.timeout_ns};

  if (warp == kBwdComputeWarps) {
    // ------------------------------------------------ producer: Q, dO once; K_0, V_0, K_1, ...
    // (Q, dO and the first S ring tiles were issued before the set-up barrier)
    if (lane == 0) {
      bool ok = true;
      for (int u = issued; u < 2 * n_kv; ++u) {
        const int s = u % S, use = u / S;
        prefetch(u + C::kPrefetchAhead);
        if (use > 0 && !w.wait(bar(kBarEmpty + s), (use - 1) & 1)) { ok = false; break; }
        issued = u + 1;
        if (p.withhold && u == 1) continue;  // test hook: V_0 is never loaded
        load_ring(u);
      }
      if (!ok) {
        w.drain(bar(kBarQ), 0);
        for (int v = issued - S > 0 ? issued - S : 0; v < issued; ++v)
          if (!(p.withhold && v == 1)) w.drain(bar(kBarFull + v % S), (v / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kBwdComputeWarps + 1) {
    // ------------------------------------------------ MMA issuer
    const uint64_t desc_q = ptx::smem_desc_sw128(sbase, 16, 1024);
    const uint64_t desc_do = ptx::smem_desc_sw128(sbase + C::kTileBytes, 16, 1024);
    const uint64_t desc_ring_k = ptx::smem_desc_sw128(sbase + C::kQOffRing, 16, 1024);
    const uint64_t desc_ring_n = ptx::smem_desc_sw128(sbase + C::kQOffRing, C::kChunkBytes, 1024);
    constexpr uint64_t kTileStep = C::kTileBytes >> 4;
    const uint32_t t_s = tmem + C::kQColS, t_dp = tmem + C::kQColDP, t_dq = tmem + C::kQColDQ;
    // Order: S(0), dP(0), S(1); then per key tile j, once dS(j) is written: dP(j+1),
    // dQ(j) += dS(j) K_j, S(j+2) into the buffer dS(j) occupies (after dQ(j) read it: the
    // tensor pipe runs one CTA's MMAs in order).  K_j is released after dQ(j), V_j after dP(j).
    auto slot = [&](int u) { return u % S; };
    auto phase = [&](int u) { return static_cast<uint32_t>((u / S) & 1); };
    auto issue_s = [&](int j) -> bool {  // S(j) = Q K_j^T into buffer j % 2
      if (!__all_sync(0xffffffffu, w.wait(bar(kBarFull + slot(2 * j)), phase(2 * j)))) return false;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        bwd_mma_nt<D>(t_s + (j & 1) * 128, desc_q, desc_ring_k + slot(2 * j) * kTileStep);
        ptx::tc_commit(bar(kBarS + (j & 1)));
      }
      __syncwarp();
      return true;
    };
    auto issue_dp = [&](int j) -> bool {  // dP(j) = dO V_j^T
      if (!__all_sync(0xffffffffu, w.wait(bar(kBarFull + slot(2 * j + 1)), phase(2 * j + 1)))) return false;
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        bwd_mma_nt<D>(t_dp, desc_do, desc_ring_k + slot(2 * j + 1) * kTileStep);
        ptx::tc_commit(bar(kBarDP));
        ptx::tc_commit(bar(kBarEmpty + slot(2 * j + 1)));  // V_j: read by this product only
      }
      __syncwarp();
      return true;
    };
    bool ok = __all_sync(0xffffffffu, w.wait(bar(kBarQ), 0));
    ptx::tc_fence_after();
    if (ok && n_kv > 0) ok = issue_s(0) && issue_dp(0) && (n_kv < 2 || issue_s(1));
    for (int j = 0; ok && j < n_kv; ++j) {
      ptx::named_barrier(kNbDS, kHandOffThreads);  // dS(j) written
      ptx::tc_fence_after();
      if (j + 1 < n_kv && !(ok = issue_dp(j + 1))) break;
      if (ptx::elect_one()) {
        bwd_mma_tn<D>(t_dq, t_s + (j & 1) * 128, desc_ring_n + slot(2 * j) * kTileStep, j > 0);  // dQ += dS K
        ptx::tc_commit(bar(kBarEmpty + slot(2 * j)));  // K_j
        if (j + 1 == n_kv) ptx::tc_commit(bar(kBarFinal));
      }
      __syncwarp();
      if (j + 2 < n_kv && !(ok = issue_s(j + 2))) break;
    }
    if (ptx::elect_one()) ptx::tc_commit(bar(kBarDrain));
    __syncwarp();
    w.drain(bar(kBarDrain), 0);
    __syncwarp();
  } else {
    // ------------------------------------------------ compute: thread = query row, warp = column half
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int qpos = qrow % p.N;
    const float neg = row_valid ? -lse_row * 1.4426950408889634f : 0.f;  // -LSE in log2 units
    const float neg_drow = row_valid ? -d_row : 0.f;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s0 = tmem + lane_off + C::kQColS + half * 64, t_dp = tmem + lane_off + C::kQColDP + half * 64;
    const float c2 = p.scale_log2;
    bool ok = true;
    int j = 0;
    for (; ok && j < n_kv; ++j) {
      const uint32_t t_s = t_s0 + (j & 1) * 128;
      ok = __all_sync(0xffffffffu, w.wait(bar(kBarS + (j & 1)), (j >> 1) & 1));
      if (!ok) break;
      ptx::tc_fence_after();
      // this row's keys in tile j: [0, lim) (past the end, and after the query when causal)
      int lim = p.N - j * 128;
      if (p.causal && qpos - j * 128 + 1 < lim) lim = qpos - j * 128 + 1;
      if (!row_valid) lim = 0;
      lim -= half * 64;  // relative to this warp's first column
      float pr[64];
      {
        uint32_t ra[32], rb[32];
        ptx::tmem_ld32x2(t_s, ra, t_s + 32, rb);
        const float2 c2v = make_float2(c2, c2), negv = make_float2(neg, neg);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(i < 32 ? ra[i] : rb[i - 32]),
                                                  __uint_as_float(i < 32 ? ra[i + 1] : rb[i - 31])), c2v, negv);
          const float e0 = ptx::ex2_approx(x.x), e1 = ptx::ex2_approx(x.y);
          pr[i] = i < lim ? e0 : 0.f;
          pr[i + 1] = i + 1 < lim ? e1 : 0.f;
        }
      }
      ok = __all_sync(0xffffffffu, w.wait(bar(kBarDP), j & 1));
      if (!ok) break;
      ptx::tc_fence_after();
      bwd_ds<false>(t_dp, t_s, pr, nullptr, neg_drow);  // dS over the S columns just read
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      ptx::named_barrier_arrive(kNbDS, kHandOffThreads);  // dS(j) handed over
    }
    // after a failed wait: the remaining arrivals, each once dP of its step is complete
    for (; j < n_kv && w.drain(bar(kBarDP), j & 1); ++j) ptx::named_barrier_arrive(kNbDS, kHandOffThreads);
    if (ok && n_kv > 0) ok = __all_sync(0xffffffffu, w.wait(bar(kBarFinal), 0));
    if (ok && n_kv > 0) {
      ptx::tc_fence_after();
      const uint32_t t_acc[1] = {tmem + lane_off + C::kQColDQ};
      const uint32_t dst[1] = {sbase};  // Q's buffer
      const float mul[1] = {p.scale};
      bwd_accs_to_smem<D, 1>(t_acc, dst, mul, row, half * (D / 2));
      ptx::fence_proxy_async_smem();
    }
    ptx::named_barrier(1, 32 * kBwdComputeWarps);
    if (ok && n_kv > 0 && threadIdx.x == 0) {
      for (int c = 0; c < C::kChunks; ++c) ptx::tma_store_3d(&tm_dq, sbase + c * C::kChunkBytes, c * 64, qt * 128, bh);
      ptx::bulk_commit();
      ptx::bulk_wait_read<0>();  // the store has read its staging: the CTA may exit
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdComputeWarps + 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  // Launched as a dependent of the dK/dV grid, this grid may start before that one ends; a CTA
  // leaves only once it has completed, so the end of this grid is the end of the backward
  // for whatever the stream runs next.
  if (threadIdx.x == 0) ptx::griddep_wait();
}

// ==================================================================== host side
namespace {

std::mutex g_bwd_dev_mutex;
int g_bwd_dev_state[kMaxDevices];  // 0 unknown, 1 ready, -1 wrong arch

// Architecture check and the backward kernels' shared-memory limits, once per device.
int prepare_device_bwd() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_bwd_dev_mutex);
  if (g_bwd_dev_state[dev] == 1) return FA_OK;
  if (g_bwd_dev_state[dev] == -1) return FA_ERR_ARCH;
  const int arch = check_arch(dev);
  if (arch != FA_OK) {
    if (arch == FA_ERR_ARCH) g_bwd_dev_state[dev] = -1;
    return arch;
  }
  if (cudaFuncSetAttribute(fa_bwd_dkdv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<64>::kSmemKV) != cudaSuccess ||
      cudaFuncSetAttribute(fa_bwd_dkdv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<128>::kSmemKV) != cudaSuccess ||
      cudaFuncSetAttribute(fa_bwd_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<64>::kSmemQ) != cudaSuccess ||
      cudaFuncSetAttribute(fa_bwd_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<128>::kSmemQ) != cudaSuccess)
    return FA_ERR_CUDA;
  g_bwd_dev_state[dev] = 1;
  return FA_OK;
}

struct BwdProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* delta;
  int B, Hq, Hkv, N, d;
  float scale;
  int causal;
};

int validate_bwd(const BwdProblem& pr) {
  const void* in[6] = {pr.q, pr.k, pr.v, pr.o, pr.lse, pr.dout};
  const void* out[4] = {pr.dq, pr.dk, pr.dv, pr.delta};
  for (const void* ptr : in)
    if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 15u)) return FA_ERR_ARG;
  for (const void* ptr : out)
    if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 15u)) return FA_ERR_ARG;
  if (pr.B < 1 || pr.Hq < 1 || pr.Hkv < 1 || pr.N < 1 || (pr.d != 64 && pr.d != 128)) return FA_ERR_ARG;
  if (pr.Hq % pr.Hkv != 0) return FA_ERR_ARG;
  if (!(pr.scale > 0.f) || !std::isfinite(pr.scale)) return FA_ERR_ARG;
  const long long q_rows = static_cast<long long>(pr.B) * pr.Hq * pr.N;
  const long long kv_rows = static_cast<long long>(pr.B) * pr.Hkv * pr.N;
  if (q_rows > 2147483647LL) return FA_ERR_ARG;
  const size_t qb = static_cast<size_t>(q_rows) * pr.d * 2, kb = static_cast<size_t>(kv_rows) * pr.d * 2;
  const size_t lb = static_cast<size_t>(q_rows) * 4;
  const size_t in_n[6] = {qb, kb, kb, qb, lb, qb};
  const size_t out_n[4] = {qb, kb, kb, lb};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(out[i], out_n[i], in[j], in_n[j])) return FA_ERR_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(out[i], out_n[i], out[j], out_n[j])) return FA_ERR_ARG;
  }
  for (const void* ptr : in)
    if (!is_device_pointer(ptr)) return FA_ERR_ARG;
  for (const void* ptr : out)
    if (!is_device_pointer(ptr)) return FA_ERR_ARG;
  return FA_OK;
}

template <int D>
int launch_bwd(const BwdProblem& pr, int withhold, unsigned long long timeout_ns, cudaStream_t stream) {
  const int G = pr.Hq / pr.Hkv;
  const int groups = pr.B * pr.Hkv;
  const int R = G * pr.N;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!encode_map(&mq, pr.q, groups, R, D) || !encode_map(&mk, pr.k, groups, pr.N, D) ||
      !encode_map(&mv, pr.v, groups, pr.N, D) || !encode_map(&mdo, pr.dout, groups, R, D) ||
      !encode_map(&mdq, pr.dq, groups, R, D) || !encode_map(&mdk, pr.dk, groups, pr.N, D) ||
      !encode_map(&mdv, pr.dv, groups, pr.N, D))
    return FA_ERR_LAUNCH;
  BwdParams p{};
  p.lse = pr.lse;
  p.dvec = pr.delta;
  p.groups = groups;
  p.R = R;
  p.N = pr.N;
  p.n_qtiles = (R + 127) / 128;
  p.n_ktiles = (pr.N + 127) / 128;
  p.scale = pr.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(pr.scale) * 1.4426950408889634);
  p.causal = pr.causal ? 1 : 0;
  p.withhold = withhold;
  p.timeout_ns = timeout_ns;
  const long long rows = static_cast<long long>(groups) * R;
  constexpr long long kRowsPerBlock = static_cast<long long>(kPrepThreads / 32) * prep_rows_per_warp<D>();
  const long long prep_blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long grid_kv = static_cast<long long>(groups) * p.n_ktiles;
  const long long grid_q = static_cast<long long>(groups) * p.n_qtiles;
  if (prep_blocks > 2147483647LL || grid_kv > 2147483647LL || grid_q > 2147483647LL) return FA_ERR_ARG;
  fa_bwd_prep_kernel<D><<<static_cast<unsigned>(prep_blocks), kPrepThreads, 0, stream>>>(
      static_cast<const uint16_t*>(pr.o), static_cast<const uint16_t*>(pr.dout), pr.delta, static_cast<int>(rows));
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  fa_bwd_dkdv_kernel<D><<<static_cast<unsigned>(grid_kv), kBwdThreads, BwdCfg<D>::kSmemKV, stream>>>(
      mq, mk, mv, mdo, mdk, mdv, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  // programmatic dependent launch: the dQ CTAs, which read nothing the dK/dV kernel writes,
  // take the SMs the dK/dV grid leaves idle in its last wave
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid_q));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = BwdCfg<D>::kSmemQ;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fa_bwd_dq_kernel<D>, mq, mk, mv, mdo, mdq, p) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

int run_bwd(const BwdProblem& pr, int withhold, unsigned long long timeout_ns, cudaStream_t stream) {
  int rc = validate_bwd(pr);
  if (rc != FA_OK) return rc;
  rc = prepare_device_bwd();
  if (rc != FA_OK) return rc;
  return pr.d == 64 ? launch_bwd<64>(pr, withhold, timeout_ns, stream)
                    : launch_bwd<128>(pr, withhold, timeout_ns, stream);
}

// ---- pipelined host-to-host backward (fa_bwd_host): chunks of K/V groups, each chunk's six
// inputs copied in on the library's copy stream, its three kernels on one of two compute
// streams, and its dQ, dK, dV copied out on the second copy stream while later chunks load and
// run.  A chunk's kernels are fa_bwd's on those groups, so the results are fa_bwd's.
struct BwdHost {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
};

int run_bwd_host(const BwdHost& h, const BwdProblem& pr, int groups_per_chunk, cudaStream_t stream) {
  int rc = validate_bwd(pr);
  if (rc != FA_OK) return rc;
  const void* hin[6] = {h.q, h.k, h.v, h.o, h.lse, h.dout};
  const void* hout[3] = {h.dq, h.dk, h.dv};
  for (const void* ptr : hin)
    if (!ptr) return FA_ERR_ARG;
  for (const void* ptr : hout)
    if (!ptr) return FA_ERR_ARG;
  if (groups_per_chunk < 0) return FA_ERR_ARG;
  const int G = pr.Hq / pr.Hkv, groups = pr.B * pr.Hkv;
  const size_t R = static_cast<size_t>(G) * pr.N;  // query rows per group
  const size_t row_bytes = static_cast<size_t>(pr.d) * 2;
  const size_t qb = groups * R * row_bytes, kb = static_cast<size_t>(groups) * pr.N * row_bytes;
  const size_t lb = groups * R * 4;
  const size_t hin_n[6] = {qb, kb, kb, qb, lb, qb};
  const size_t hout_n[3] = {qb, kb, kb};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(hout[i], hout_n[i], hin[j], hin_n[j])) return FA_ERR_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(hout[i], hout_n[i], hout[j], hout_n[j])) return FA_ERR_ARG;
  }
  for (const void* ptr : hin)
    if (!is_pinned_host(ptr)) return FA_ERR_ARG;
  for (const void* ptr : hout)
    if (!is_pinned_host(ptr)) return FA_ERR_ARG;
  rc = prepare_device_bwd();
  if (rc != FA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe[dev].mu);
  HostPipe* hp = nullptr;
  rc = host_pipe(dev, &hp);
  if (rc != FA_OK) return rc;
  // chunk starts need no alignment beyond a row: Q-like and K-like rows are 128 or 256 bytes,
  // and the kernels read LSE and D one float per row
  int sizes[kMaxChunks];
  const double bytes = 5.0 * qb + 4.0 * kb + lb;  // in: q, k, v, o, lse, dO; out: dq, dk, dv
  const double flops = 10.0 * static_cast<double>(pr.B) * pr.Hq * pr.N * pr.N * pr.d * (pr.causal ? 0.5 : 1.0);
  const int n_chunks = chunk_sizes(groups, groups_per_chunk, bytes, flops / kBackwardFlopsPerSec, sizes);
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
    const size_t k_off = static_cast<size_t>(g0) * pr.N * row_bytes, k_len = static_cast<size_t>(ng) * pr.N * row_bytes;
    const size_t l_off = g0 * R * 4, l_len = ng * R * 4;
    const struct { void* dst; const void* src; size_t off, len; } in[6] = {
        {const_cast<void*>(pr.q), h.q, q_off, q_len},       {const_cast<void*>(pr.k), h.k, k_off, k_len},
        {const_cast<void*>(pr.v), h.v, k_off, k_len},       {const_cast<void*>(pr.o), h.o, q_off, q_len},
        {const_cast<float*>(pr.lse), h.lse, l_off, l_len},  {const_cast<void*>(pr.dout), h.dout, q_off, q_len}};
    for (const auto& x : in)
      if (cudaMemcpyAsync(at_mut(x.dst, x.off), at(x.src, x.off), x.len, cudaMemcpyHostToDevice, hp->in) != cudaSuccess)
        return FA_ERR_CUDA;
    cudaStream_t cs = hp->comp[c % kComputeStreams];
    if (cudaEventRecord(hp->loaded[c], hp->in) != cudaSuccess || cudaStreamWaitEvent(cs, hp->loaded[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    BwdProblem sub = pr;
    sub.q = at(pr.q, q_off);
    sub.k = at(pr.k, k_off);
    sub.v = at(pr.v, k_off);
    sub.o = at(pr.o, q_off);
    sub.lse = reinterpret_cast<const float*>(at(pr.lse, l_off));
    sub.dout = at(pr.dout, q_off);
    sub.dq = at_mut(pr.dq, q_off);
    sub.dk = at_mut(pr.dk, k_off);
    sub.dv = at_mut(pr.dv, k_off);
    sub.delta = reinterpret_cast<float*>(at_mut(pr.delta, l_off));
    sub.B = 1;
    sub.Hq = ng * G;
    sub.Hkv = ng;
    rc = pr.d == 64 ? launch_bwd<64>(sub, 0, kDefaultTimeoutNs, cs) : launch_bwd<128>(sub, 0, kDefaultTimeoutNs, cs);
    if (rc != FA_OK) return rc;
    if (cudaEventRecord(hp->computed[c], cs) != cudaSuccess || cudaStreamWaitEvent(hp->out, hp->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.dq, q_off), at(pr.dq, q_off), q_len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.dk, k_off), at(pr.dk, k_off), k_len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess ||
        cudaMemcpyAsync(at_mut(h.dv, k_off), at(pr.dv, k_off), k_len, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  if (cudaEventRecord(hp->done, hp->out) != cudaSuccess || cudaStreamWaitEvent(stream, hp->done, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

int bwd_status_word(int clear) {
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

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, float* delta, int B, int Hq, int Hkv, int N, int d, float scale,
           int causal, cudaStream_t stream) {
  const fa::BwdProblem pr{q, k, v, o, lse, dout, dq, dk, dv, delta, B, Hq, Hkv, N, d, scale, causal};
  return fa::run_bwd(pr, 0, fa::kDefaultTimeoutNs, stream);
}

int fa_bwd_host(const void* q_host, const void* k_host, const void* v_host, const void* o_host,
                const float* lse_host, const void* dout_host, void* dq_host, void* dk_host, void* dv_host,
                void* q, void* k, void* v, void* o, float* lse, void* dout, void* dq, void* dk, void* dv,
                float* delta, int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                int groups_per_chunk, cudaStream_t stream) {
  const fa::BwdProblem pr{q, k, v, o, lse, dout, dq, dk, dv, delta, B, Hq, Hkv, N, d, scale, causal};
  const fa::BwdHost h{q_host, k_host, v_host, o_host, lse_host, dout_host, dq_host, dk_host, dv_host};
  return fa::run_bwd_host(h, pr, groups_per_chunk, stream);
}

int fa_bwd_withheld_tile(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int Hq, int Hkv,
                         int N, int d, float scale, int causal, double wait_timeout_ms, cudaStream_t stream) {
  if (!(wait_timeout_ms >= 1.0 && wait_timeout_ms <= 10000.0)) return FA_ERR_ARG;
  const fa::BwdProblem pr{q, k, v, o, lse, dout, dq, dk, dv, delta, B, Hq, Hkv, N, d, scale, causal};
  return fa::run_bwd(pr, 1, static_cast<unsigned long long>(wait_timeout_ms * 1e6), stream);
}

}  // extern "C"
