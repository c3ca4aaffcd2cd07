// Newton-Schulz products on the 5th-generation tensor cores.
//
// One iteration of the Muon orthogonalisation ("How to train a GPT model in
// 3 minutes", section 2, custom Muon optimizer: a Newton-Schulz iteration in
// place of an SVD) is X <- a X + (b A + c A A) X with A = X X^T. Two kernels
// carry it, both instances of the template below:
//
//   Gram     (kGram = true):  out = s_acc * (Y Y^T) + s_e * E, Y an n x K
//            matrix read through one K-major tensor map. Tiles are 128 rows x
//            256 columns; only tiles that reach the upper triangle are
//            computed (tile row I <= 2J + 1 for tile column J), and the
//            epilogue writes each 128 x 128 block above the diagonal in place
//            and transposed, so the n x n output is full.
//            With Y = X and s_acc = b it produces B = b A directly (c = 0).
//            With Y = A (symmetric, so A A = A A^T), s_acc = c, E = A and
//            s_e = b it produces B = b A + c A A.
//   Combine  (kGram = false): out = s_acc * (B X) + s_e * E with B K-major
//            (n x n) and X MN-major (n x m, row-major): E = X, s_e = a gives
//            X' = a X + B X with the combination done on the fp32
//            accumulator before the single bf16 rounding. Under the precise
//            carry E and X' are each a pair of bf16 parts (hi + lo); the last
//            combine can write the caller's matrices directly (FinalArgs).
//
// Structure: a persistent grid of 2-CTA clusters (one CTA per SM) walks a
// host-built tile list covering every matrix of every shape group in the
// batch. The pair runs paired-SM MMAs (tcgen05 cta_group::2, M = 256): each
// CTA owns 128 rows of a 256 x 256 output tile and loads its own A rows and
// its own half of B; no load is shared between the two CTAs. Warp 0 issues TMA
// loads into a ring of shared-memory stages, one thread of warp 1 of the even
// CTA issues tcgen05.mma into a double-buffered fp32 accumulator in tensor
// memory of both CTAs, and warps 2-9 drain the accumulator (tcgen05.ld), apply the
// epilogue and store bf16 to global memory by TMA. A host-built schedule gives
// each cluster its own list of tiles, balanced by contraction length. Every
// wait is bounded (see mbar_wait_bounded).
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace muon {

constexpr int kMaxGroups = 6;   // shape groups served by one launch
constexpr int kGemmThreads = 320;  // producer warp, MMA warp, 8 epilogue warps
constexpr int kEpilogueThreads = 256;

struct GemmGroup {
  const uint16_t* e;      // non-null when the epilogue adds s_e * E (E read through map_e)
  const float* post;      // per-matrix scale of this launch's operand X (nullptr: 1); the Gram
                          // output takes post^2, the combine output post (X0 left unscaled)
  int64_t mat_stride;     // elements between consecutive matrices of e
  int rows_out, cols_out, ld_out;
  int nk;                 // number of 64-wide k-blocks of the contraction
};

struct GemmArgs {
  CUtensorMap map_a[kMaxGroups];  // operand A: K-major, box 64 x 128
  CUtensorMap map_b[kMaxGroups];  // operand B: Gram: same as A; combine: MN-major, box 64 x 64
  CUtensorMap map_out[kMaxGroups];     // output, box 64 columns x 128 rows, 128-byte swizzle
  CUtensorMap map_mirror[kMaxGroups];  // Gram output again, box 128 columns x 64 rows, no swizzle
  CUtensorMap map_e[kMaxGroups];       // addend E, box 64 columns x 128 rows, 128-byte swizzle
  // Combine under the precise carry: the low parts of E and of the output, same boxes.
  CUtensorMap map_e_lo[kMaxGroups];
  CUtensorMap map_out_lo[kMaxGroups];
  GemmGroup grp[kMaxGroups];
  const int4* tiles;              // {group, matrix within group, tile row, tile col}
  const int* cta_begin;           // CTA b walks tiles[cta_begin[b] .. cta_begin[b+1])
  int num_tiles;
  int grid;                       // CTAs launched (entries of cta_begin minus one)
  int num_groups;
  float s_acc;
  float s_e;
  int* err;
  unsigned long long* clk;  // non-null while profiling: += {SM cycles, ns} of every CTA of the launch
  int carry;                // combine: X is carried as hi + lo (E and the output each in two bf16 parts)
};

// The last combine of a call can write its result straight into the caller's
// bf16 matrices: W <- W - scale * X_k (muon_step) or out <- X_k
// (muon_orthogonalize). One tensor map per matrix, in the order
// first[group] + matrix-within-group: box 64 columns x 128 rows, 128-byte
// swizzle; or, with trans = 1 (the caller's matrix is X_k^T, rows > cols),
// 128 columns x 64 rows, unswizzled, and the tile's values go in transposed.
constexpr int kMaxFinal = 160;

template <int N>
struct FinalArgs {
  CUtensorMap map[N];
  float scale[N];
  uint8_t trans[N];
  int first[kMaxGroups];
  int update;  // 1: W <- keep * W - scale * X_k; 0: out <- X_k
  float keep;  // 1 - lr * weight_decay
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Waits that must not be cut short by the abort flag: used only to let copies
// and MMAs already in flight land before the CTA releases its resources.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}

template <bool kGram, int kBN, int kStages>
struct GemmShape {
  static constexpr int BM = 128;
  static constexpr int BK = 64;
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  // Paired-SM MMAs: each CTA holds only its half of B's columns.
  static constexpr uint32_t B_BYTES = (kBN / 2) * BK * 2;
  static constexpr uint32_t TMEM_COLS = 2 * kBN;
  static constexpr uint32_t STAGING_BYTES = 4 * 16384;  // two 128 x 64 bf16 boxes per column half
  static constexpr uint32_t BAR_BYTES = 8 * (2 * kStages + 5 + 4) + 16;  // + one barrier per staging box
  // 1024 bytes of slack to align the swizzled tiles to 1024.
  static constexpr uint32_t SMEM_BYTES = 1024 + kStages * (A_BYTES + B_BYTES) + STAGING_BYTES + BAR_BYTES;
};

// The two CTAs of a cluster take tile rows I and I+1 of the same tile column,
// so they need the same B block. Paired-SM MMAs (tcgen05 cta_group::2,
// M = 256): each CTA loads its own A rows and its own half of B's columns into
// its own shared memory, signalling the even (leader) CTA's full barrier; the
// leader's single MMA thread issues M = 256 MMAs that read both CTAs' shared
// memory and write each CTA's 128 accumulator rows into its own TMEM. Commits
// arrive on the barrier at the same offset in both CTAs; the odd CTA's
// epilogue releases the accumulator on the leader's barrier.
constexpr int kCluster = 2;

template <bool kGram, int kBN, int kStages, bool kFinal>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_gemm_kernel(const __grid_constant__ GemmArgs args, const __grid_constant__ FinalArgs<kFinal ? kMaxFinal : 1> fin) {
  using S = GemmShape<kGram, kBN, kStages>;
  constexpr int BM = S::BM, BK = S::BK;
  constexpr uint32_t A_BYTES = S::A_BYTES, B_BYTES = S::B_BYTES;
  constexpr uint32_t kIdesc = instr_desc_bf16(2 * BM, kBN, !kGram);
  constexpr uint16_t kPairMask = 0x3;
  static_assert(kBN == 256, "tile width");
  static_assert(!(kGram && kFinal), "only the combine writes to the caller's matrices");
  static_assert(S::TMEM_COLS == 512, "TMEM allocation must be a power of two");

  const long long clk_start = clock64();
  const uint64_t ns_start = global_timer_ns();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * A_BYTES;
  uint8_t* staging = sB + kStages * B_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + S::STAGING_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5 + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_cta_rank());
  const int list = blockIdx.x / kCluster;  // this cluster's tile list
  const int t_begin = args.cta_begin[list], t_end = args.cta_begin[list + 1];
  const uint32_t bar0 = smem_u32(bars);
  // full[s]: stage s loaded; empty[s]: stage s consumed by the MMAs (of both CTAs);
  // tfull[a]: accumulator a complete; tempty[a]: accumulator a drained; drain: abort path.
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (kStages + st); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
  auto addend_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };  // staging box i's TMA load

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      // One arrival per epilogue warp of both CTAs, on the leader's barrier.
      mbar_init(tempty_bar(a), 2 * (kEpilogueThreads / 32));
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(addend_bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < args.num_groups; ++g) {
      tma_prefetch_map(&args.map_a[g]);
      tma_prefetch_map(&args.map_b[g]);
      if (!kFinal) tma_prefetch_map(&args.map_out[g]);
      if (kGram) tma_prefetch_map(&args.map_mirror[g]);
      if (args.grp[g].e) tma_prefetch_map(&args.map_e[g]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), S::TMEM_COLS);  // with warp 1 of the peer CTA
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anything is sent to them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above overlaps the previous kernel's tail; its outputs are read only below.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;        // bit s: stage s has a load in flight or landed
      uint32_t armed_parity = 0; // bit s: parity of that load's phase
      for (int t = t_begin; t < t_end; ++t) {
        const int4 td = args.tiles[t];
        const int I = td.z + rank;
        const GemmGroup& G = args.grp[td.x];
        const CUtensorMap* ma = &args.map_a[td.x];
        const CUtensorMap* mb = &args.map_b[td.x];
        // Gram tiles whose 128 A rows lie inside the 256-row B block read A from B's copy.
        const bool a_in_b = kGram && ((I >> 1) == td.w);
        const uint32_t bytes = a_in_b ? B_BYTES : A_BYTES + B_BYTES;
        bool ok = true;
        for (int kb = 0; kb < G.nk; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) {
            ok = false;
            break;
          }
          // Both CTAs' loads complete on the leader's full barrier, which expects them all.
          const uint32_t leader_full = mapa_shared(full_bar(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * bytes);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (!a_in_b)
            tma_load_3d_pair(smem_u32(sA + stage * A_BYTES), ma, leader_full, kb * BK, I * BM, td.y);
          const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
          if (kGram) {  // this CTA's 128 of the 256 B rows
            tma_load_3d_pair(b_dst, mb, leader_full, kb * BK, td.w * kBN + rank * 128, td.y);
          } else {      // this CTA's 128 of the 256 B columns, two boxes of 64
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_3d_pair(b_dst + c * 8192u, mb, leader_full, td.w * kBN + rank * 128 + c * 64, kb * BK, td.y);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag && rank == 0) {
        // Let loads already issued land before the CTA's shared memory is released.
        for (int st = 0; st < kStages; ++st)
          if (armed & (1u << st)) mbar_wait_drain(full_bar(st), (armed_parity >> st) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool issued = false;
      for (int t = t_begin; t < t_end; ++t) {
        const int4 td = args.tiles[t];
        const int I = td.z + rank;
        const int nk = args.grp[td.x].nk;
        const bool a_in_b = kGram && ((I >> 1) == td.w);
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
          // Each CTA's B half holds its own 128 rows, so an A inside B is the whole half.
          const uint32_t a_addr = a_in_b ? b_addr : smem_u32(sA + stage * A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // K-major: the next 16 k-values are 32 bytes further along each 128-byte row.
            const uint64_t a_desc = smem_desc_sw128(a_addr + k * 32u, 16u, 1024u);
            // MN-major: the next 16 k-values are 16 rows (2048 bytes) further down.
            const uint64_t b_desc = kGram ? smem_desc_sw128(b_addr + k * 32u, 16u, 1024u)
                                          : smem_desc_sw128(b_addr + k * 2048u, 8192u, 1024u);
            mma_bf16_ss_pair(d_tmem, a_desc, b_desc, kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit_pair_multicast(empty_bar(stage), kPairMask);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_multicast(tfull_bar(acc), kPairMask);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (*abort_flag && issued) {
        mma_commit_pair_multicast(drain_bar, 0x1);
        mbar_wait_drain(drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Eight warps, two per TMEM lane quarter. The four warps of a column half work together on
    // 128-row x 64-column boxes: each writes its 32 rows into a shared staging box, and one thread
    // moves the whole 16 KB box with a single TMA operation (addend load, output store, mirrored
    // store). A half owns two staging boxes; both of a tile's addend loads are in flight before
    // its accumulator is ready, and a box is rewritten only once the store issued from it has
    // read it. Named barrier 1 + half keeps the four warps in step.
    constexpr int kHalfCols = kBN / 2;
    constexpr int kBoxes = kHalfCols / 64;
    static_assert(kBoxes == 2, "one staging box per 64 columns of a half");
    const int quarter = warp & 3;  // TMEM lanes this warp may read: 32*quarter .. +31
    const int half = (warp - 2) >> 2;
    const bool leader = quarter == 0 && lane == 0;  // issues the half's TMA operations
    const uint32_t half_bar = 1u + static_cast<uint32_t>(half);
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    uint8_t* const stg_base = staging + half * 32768;
    const uint32_t bar_base = addend_bar(2 * half);
    uint32_t box_phase = 0u;    // bit b
    uint32_t box_pending = 0u;  // bit b: a load into box b was issued and not yet waited for
    auto stg_box = [&](int b) { return stg_base + b * 16384; };
    auto box_bar = [&](int b) { return bar_base + 8u * static_cast<uint32_t>(b); };
    auto sync_half = [&]() { named_barrier_sync(half_bar, 128); };
    // Loads a 16 KB box into staging box b by TMA, once earlier stores have read it (leader).
    auto load_box = [&](int b, const CUtensorMap* map, int x, int y, int z, bool wait_all) {
      if (leader) {
        if (wait_all)
          bulk_wait_group_read0();
        else
          bulk_wait_group_read<1>();
        mbar_arrive_expect_tx(box_bar(b), 16384u);
        tma_load_3d(smem_u32(stg_box(b)), map, box_bar(b), x, y, z);
      }
      box_pending |= 1u << b;
    };
    auto wait_box = [&](int b) -> bool {
      if (!mbar_wait_bounded(box_bar(b), (box_phase >> b) & 1u, abort_flag, args.err)) return false;
      box_phase ^= 1u << b;
      box_pending &= ~(1u << b);
      return true;
    };
    // Box b has been written by all four warps: the leader stores it through `map` at (x, y, z).
    auto store_box = [&](int b, const CUtensorMap* map, int x, int y, int z) {
      fence_proxy_async_smem();
      sync_half();
      if (leader) {
        tma_store_3d(map, smem_u32(stg_box(b)), x, y, z);
        bulk_commit_group();
      }
    };
    // Box b may be overwritten once the store issued from it has read it: the leader waits, all
    // four warps meet (`pending`: stores allowed to be still reading, the newest first).
    auto free_box = [&](bool all) {
      if (leader) {
        if (all)
          bulk_wait_group_read0();
        else
          bulk_wait_group_read<1>();
      }
      sync_half();
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    int ring = 0;  // Gram: staging boxes are used in turn by every store
    const bool carry = !kGram && args.carry != 0;
    // Precise carry: box 0 holds the high part and box 1 the low part of unit u's addend. v gets
    // s_e * (hi + lo) added, and the two boxes then take the output's high and low parts in place.
    auto add_carried_addend = [&](float (&v)[64], float s_e_) {
      wait_box(0);
      wait_box(1);
      const uint8_t* rh = stg_box(0) + (quarter * 32 + lane) * 128;
      const uint8_t* rl = stg_box(1) + (quarter * 32 + lane) * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 h4 = *reinterpret_cast<const uint4*>(rh + ((j ^ (lane & 7)) * 16));
        const uint4 l4 = *reinterpret_cast<const uint4*>(rl + ((j ^ (lane & 7)) * 16));
        const uint32_t hh[4] = {h4.x, h4.y, h4.z, h4.w}, ll[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          v[8 * j + 2 * h] += s_e_ * (bf16_bits_to_float(hh[h] & 0xFFFFu) + bf16_bits_to_float(ll[h] & 0xFFFFu));
          v[8 * j + 2 * h + 1] += s_e_ * (bf16_bits_to_float(hh[h] >> 16) + bf16_bits_to_float(ll[h] >> 16));
        }
      }
    };
    for (int t = t_begin; t < t_end; ++t) {
      const int4 td = args.tiles[t];
      const int I = td.z + rank;
      const GemmGroup& G = args.grp[td.x];
      const bool has_e = G.e != nullptr;
      // Gram: this half is the 128x128 block (tile row I, block column 2*td.w + half). Blocks
      // below the diagonal are skipped (their transposes come from other tiles), blocks above it are
      // stored twice (in place and mirrored), the diagonal block once.
      const int block_col = 2 * td.w + half;
      const bool skip = kGram && (block_col < I);
      const bool mirror = kGram && (block_col > I);
      const int col_base = td.w * kBN + half * kHalfCols;
      const int y_tile = I * BM;
      // X = post * X' with X' the stored operand: the Gram gets post^2 on the product, the
      // combine post on both of its terms.
      const float post = G.post ? __ldg(G.post + td.y) : 1.0f;
      const float s_acc = args.s_acc * (kGram ? post * post : post);
      const float s_e = args.s_e * (kGram ? 1.0f : post);
      // Addend boxes (box b of this tile through staging box b): box 0 may reuse its staging box
      // once all but the latest store have read theirs, box 1 once all have.
      // Under the precise carry the two boxes hold the high and low parts of one unit's addend,
      // and both wait until every store has read its box.
      if (has_e && !skip) {
        if (carry) {
          load_box(0, &args.map_e[td.x], col_base, y_tile, td.y, true);
          load_box(1, &args.map_e_lo[td.x], col_base, y_tile, td.y, true);
        } else {
          load_box(0, &args.map_e[td.x], col_base, y_tile, td.y, false);
          load_box(1, &args.map_e[td.x], col_base + 64, y_tile, td.y, true);
        }
      }
      // A wait that gives up (and raises the CTA abort flag) does not leave the loop on its own:
      // every warp of the half goes through the same barriers, and all four leave together after
      // the end-of-tile barrier below.
      mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.err);
      tc_fence_after();
      bool released = false;  // the accumulator has been handed back to the MMA warp
      if (carry && !skip) {
        // Precise carry: the two units of the half run one after the other through both boxes.
#pragma unroll 1
        for (int box = 0; box < kBoxes; ++box) {
          const int x0 = col_base + box * 64;
          if (box == 1) {  // unit 1's addend parts, once every store has read its box
            load_box(0, &args.map_e[td.x], x0, y_tile, td.y, true);
            load_box(1, &args.map_e_lo[td.x], x0, y_tile, td.y, true);
          }
          float v[64];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
            tmem_load_32cols(
                tmem_base + lane_field + static_cast<uint32_t>(acc * kBN + half * kHalfCols + box * 64 + cc * 32), r);
            tmem_load_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[cc * 32 + k] = s_acc * __uint_as_float(r[k]);
          }
          add_carried_addend(v, s_e);
          uint8_t* rh = stg_box(0) + (quarter * 32 + lane) * 128;
          uint8_t* rl = stg_box(1) + (quarter * 32 + lane) * 128;
          if constexpr (kFinal) {
            // X_k = v exactly as carried: W' = keep * W - scale * X_k, or out = bf16(X_k), through box 0.
            const int mi = fin.first[td.x] + td.y;
            const bool tr = fin.trans[mi] != 0;
            const float us = fin.scale[mi];
            const int ux = tr ? y_tile : x0, uy = tr ? x0 : y_tile;
            if (fin.update) {
              fence_proxy_async_smem();  // the addend reads above come before the load's writes
              sync_half();
              if (leader) {
                mbar_arrive_expect_tx(box_bar(0), 16384u);
                tma_load_3d(smem_u32(stg_box(0)), &fin.map[mi], box_bar(0), ux, uy, 0);
              }
              box_pending |= 1u;
              wait_box(0);
            }
            if (!tr) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint4* q = reinterpret_cast<uint4*>(rh + ((j ^ (lane & 7)) * 16));
                uint32_t ww[4] = {0u, 0u, 0u, 0u};
                if (fin.update) {
                  const uint4 w4 = *q;
                  ww[0] = w4.x; ww[1] = w4.y; ww[2] = w4.z; ww[3] = w4.w;
                }
                uint32_t o[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float x0v = v[8 * j + 2 * h], x1v = v[8 * j + 2 * h + 1];
                  o[h] = fin.update ? pack_bf16x2(fin.keep * bf16_bits_to_float(ww[h] & 0xFFFFu) - us * x0v,
                                                  fin.keep * bf16_bits_to_float(ww[h] >> 16) - us * x1v)
                                    : pack_bf16x2(x0v, x1v);
                }
                *q = make_uint4(o[0], o[1], o[2], o[3]);
              }
            } else {
              uint16_t* q = reinterpret_cast<uint16_t*>(stg_box(0));
#pragma unroll
              for (int c = 0; c < 64; ++c) {
                const int idx = c * 128 + quarter * 32 + lane;
                q[idx] = fin.update ? to_bf16_bits(fin.keep * bf16_bits_to_float(q[idx]) - us * v[c]) : to_bf16_bits(v[c]);
              }
            }
            store_box(0, &fin.map[mi], ux, uy, 0);
          } else {
            // The output's high and low parts, in place of the addend's (each thread rewrites its own row).
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t oh[4], ol[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float x0v = v[8 * j + 2 * h], x1v = v[8 * j + 2 * h + 1];
                oh[h] = pack_bf16x2(x0v, x1v);
                ol[h] = pack_bf16x2(x0v - bf16_bits_to_float(oh[h] & 0xFFFFu), x1v - bf16_bits_to_float(oh[h] >> 16));
              }
              *reinterpret_cast<uint4*>(rh + ((j ^ (lane & 7)) * 16)) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
              *reinterpret_cast<uint4*>(rl + ((j ^ (lane & 7)) * 16)) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
            }
            store_box(0, &args.map_out[td.x], x0, y_tile, td.y);
            store_box(1, &args.map_out_lo[td.x], x0, y_tile, td.y);
          }
        }
      } else if constexpr (kFinal) {
        // The last combine writes straight into the caller's matrices. Both boxes of X_k are first
        // taken into registers as bf16 (the value the workspace would have held), the accumulator
        // is released at once, and only then are the caller's two boxes loaded in place of the
        // addends, both in flight together: W' = keep * W - scale * X_k, or out = X_k.
        uint32_t pk[2][32];
#pragma unroll
        for (int box = 0; box < kBoxes; ++box) {
          float v[64];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
            tmem_load_32cols(
                tmem_base + lane_field + static_cast<uint32_t>(acc * kBN + half * kHalfCols + box * 64 + cc * 32), r);
            tmem_load_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[cc * 32 + k] = s_acc * __uint_as_float(r[k]);
          }
          const uint8_t* row_ptr = stg_box(box) + (quarter * 32 + lane) * 128;
          wait_box(box);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 w4 = *reinterpret_cast<const uint4*>(row_ptr + ((j ^ (lane & 7)) * 16));
            const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
              pk[box][4 * j + h] = pack_bf16x2(v[8 * j + 2 * h] + s_e * bf16_bits_to_float(ww[h] & 0xFFFFu),
                                               v[8 * j + 2 * h + 1] + s_e * bf16_bits_to_float(ww[h] >> 16));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));  // the leader's barrier
        released = true;
        const int mi = fin.first[td.x] + td.y;
        const bool tr = fin.trans[mi] != 0;
        const float us = fin.scale[mi];
        if (fin.update) {
          fence_proxy_async_smem();  // the addend reads above come before the loads' writes
          sync_half();
#pragma unroll
          for (int box = 0; box < kBoxes; ++box) {
            const int x0 = col_base + box * 64;
            if (leader) {
              mbar_arrive_expect_tx(box_bar(box), 16384u);
              tma_load_3d(smem_u32(stg_box(box)), &fin.map[mi], box_bar(box), tr ? y_tile : x0, tr ? x0 : y_tile, 0);
            }
            box_pending |= 1u << box;
          }
        }
#pragma unroll
        for (int box = 0; box < kBoxes; ++box) {
          const int x0 = col_base + box * 64;
          if (fin.update) wait_box(box);
          if (!tr) {
            // The box at (x0, y_tile), swizzled like the addend: this thread's row, chunk j at j ^ (lane & 7).
            uint8_t* row_ptr = stg_box(box) + (quarter * 32 + lane) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4* q = reinterpret_cast<uint4*>(row_ptr + ((j ^ (lane & 7)) * 16));
              uint32_t o[4] = {pk[box][4 * j], pk[box][4 * j + 1], pk[box][4 * j + 2], pk[box][4 * j + 3]};
              if (fin.update) {
                const uint4 w4 = *q;
                const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int h = 0; h < 4; ++h)
                  o[h] = pack_bf16x2(fin.keep * bf16_bits_to_float(ww[h] & 0xFFFFu) - us * bf16_bits_to_float(o[h] & 0xFFFFu),
                                     fin.keep * bf16_bits_to_float(ww[h] >> 16) - us * bf16_bits_to_float(o[h] >> 16));
              }
              *q = make_uint4(o[0], o[1], o[2], o[3]);
            }
          } else {
            // The transposed box: 64 rows (the box's columns) x 128 columns (the tile's rows), unswizzled.
            uint16_t* q = reinterpret_cast<uint16_t*>(stg_box(box));
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int idx = c * 128 + quarter * 32 + lane;
              const uint16_t xk = static_cast<uint16_t>((c & 1) ? (pk[box][c >> 1] >> 16) : (pk[box][c >> 1] & 0xFFFFu));
              q[idx] = fin.update ? to_bf16_bits(fin.keep * bf16_bits_to_float(q[idx]) - us * bf16_bits_to_float(xk)) : xk;
            }
          }
          store_box(box, &fin.map[mi], tr ? y_tile : x0, tr ? x0 : y_tile, 0);
        }
      } else if (!skip) {
#pragma unroll
        for (int box = 0; box < kBoxes; ++box) {
          float v[64];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
            tmem_load_32cols(
                tmem_base + lane_field + static_cast<uint32_t>(acc * kBN + half * kHalfCols + box * 64 + cc * 32), r);
            tmem_load_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[cc * 32 + k] = s_acc * __uint_as_float(r[k]);
          }
          const int x0 = col_base + box * 64;
          // The staging box for this output: the addend's box, or the next in turn (Gram).
          const int b = has_e ? box : (ring & 1);
          // This thread's row of the 128 x 64 box: 16-byte chunk j at position j ^ (row & 7) = j ^ (lane & 7).
          uint8_t* row_ptr = stg_box(b) + (quarter * 32 + lane) * 128;
          if (has_e) {
            wait_box(b);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 w4 = *reinterpret_cast<const uint4*>(row_ptr + ((j ^ (lane & 7)) * 16));
              const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                v[8 * j + 2 * h] += s_e * bf16_bits_to_float(ww[h] & 0xFFFFu);
                v[8 * j + 2 * h + 1] += s_e * bf16_bits_to_float(ww[h] >> 16);
              }
            }
          } else {
            free_box(false);  // the store two back from this box has read it
            ++ring;
          }
          {
            uint32_t packed[32];  // this thread's 64 output values of the box, as bf16 pairs
#pragma unroll
            for (int k = 0; k < 32; ++k) packed[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(row_ptr + ((j ^ (lane & 7)) * 16)) =
                  make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
            store_box(b, &args.map_out[td.x], x0, y_tile, td.y);
            if (mirror) {
              // The transposed box: 64 rows (this box's columns) x 128 columns (the tile's rows),
              // unswizzled. Without an addend it goes through the next staging box in turn; with
              // one (the A A pass), the other box may still hold the next addend, so it reuses
              // this box once the store just issued from it has read it.
              int bm = b;
              if (has_e) {
                free_box(true);
              } else {
                bm = ring & 1;
                ++ring;
                free_box(false);
              }
              uint16_t* p = reinterpret_cast<uint16_t*>(stg_box(bm));
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                p[(2 * k) * 128 + quarter * 32 + lane] = static_cast<uint16_t>(packed[k] & 0xFFFFu);
                p[(2 * k + 1) * 128 + quarter * 32 + lane] = static_cast<uint16_t>(packed[k] >> 16);
              }
              store_box(bm, &args.map_mirror[td.x], y_tile, x0, td.y);
            }
          }
        }
      }
      // All four warps take the same decision, even when another warp raises the flag between their reads.
      if (named_barrier_or(half_bar, 128, *abort_flag != 0)) break;
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));  // the leader's barrier
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (leader) {
      for (int b = 0; b < 2; ++b)  // abort path: let loads land
        if ((box_pending >> b) & 1u) mbar_wait_drain(box_bar(b), (box_phase >> b) & 1u);
      bulk_wait_group0();  // every store of this half has reached global memory
    }
  }

  __syncthreads();
  // No CTA leaves while its peer may still deliver loads or MMA-commit arrivals into it.
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
  }
  if (args.clk && threadIdx.x == 0) {
    atomicAdd(args.clk, static_cast<unsigned long long>(clock64() - clk_start));
    atomicAdd(args.clk + 1, static_cast<unsigned long long>(global_timer_ns() - ns_start));
  }
}

}  // namespace muon
