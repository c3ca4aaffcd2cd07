// Every Newton-Schulz iteration of a whole batch in one persistent launch.
//
// The iteration ("How to train a GPT model in 3 minutes", section 2, custom Muon optimizer: a
// Newton-Schulz iteration in place of an SVD) is X <- a X + (b A + c A A) X with A = X X^T. For
// one matrix each iteration is a chain of stages, each a set of independent 256 x 256 output tiles:
//
//   Gram     B = b X X^T            (c = 0)   or   A = X X^T  then  B = c A A + b A   (c != 0)
//   Combine  X' = a X + B X
//
// A launch per stage (ns_gemm.cuh) leaves SMs idle at each stage's ramp and tail and between
// launches. Here one persistent grid of 2-CTA clusters runs all stages of all matrices. Each
// cluster walks its own host-built list of work items; an item is one tile of one stage of one
// matrix. A per-matrix counter in global memory counts the epilogue halves that have finished
// (four per tile: two CTAs x two column halves), and an item waits, before it reads anything the
// stage before it wrote, until the counter reaches the number of halves of all earlier stages of
// its matrix. The host orders items by a simulated list schedule (muon_api.cu) in which an item's
// result lands some time after its last MMA, and a free cluster takes, among the items that can
// start, the one with the longest chain of stages still ahead of its matrix; different matrices'
// stages then overlap each other's hand-offs.
//
// Deadlock freedom: every cluster is resident at once (the grid is the occupancy limit), every
// cluster's list is in increasing global order, and an item depends only on items earlier in that
// order. The lowest blocked item then depends only on items that are running or done, so some
// item always progresses. Every wait is bounded anyway (2 s, then MUON_ERR_TIMEOUT).
//
// Memory ordering of one dependency: the producing epilogue's TMA stores complete
// (cp.async.bulk.wait_group 0), a proxy fence orders them before a release add to the counter;
// the consumer's acquire load sees the count, and a proxy fence orders it before its TMA loads.
//
// The tile mechanics (paired-SM tcgen05 MMAs, TMA stages, staging boxes, mirrored Gram stores,
// the precise carry, the final combine into the caller's matrices) are those of ns_gemm.cuh.
#pragma once

#include "ns_gemm.cuh"

namespace muon {

enum NsItemKind : int { kNsGram = 0, kNsGramAA = 1, kNsComb = 2 };
// Tensor maps of a shape group, in global memory: [group][role].
enum NsRole : int {
  kRoleX0 = 0,    // X_0 buffer, box 64 x 128 (Gram operands, combine addend and output)
  kRoleX1 = 1,    // X_1 buffer, same
  kRoleXmn0 = 2,  // X_0 buffer, box 64 x 64 (combine B operand, MN-major)
  kRoleXmn1 = 3,
  kRoleP = 4,     // B buffer, box 64 x 128 (combine A operand, Gram and A A output)
  kRolePm = 5,    // B buffer, box 128 x 64 unswizzled (mirrored Gram stores)
  kRoleA = 6,     // A buffer (c != 0), box 64 x 128
  kRoleAm = 7,
  kRoleLo0 = 8,   // precise carry: low parts of X_0 / X_1, box 64 x 128
  kRoleLo1 = 9,
  kNumRoles = 10
};
// Item flags: first iteration (the folded scale applies), last iteration, X_t in buffer 1.
constexpr int kNsFirst = 1, kNsLast = 2, kNsOdd = 4;

struct NsGroup {
  int n, m, count, first_slot;
  int nk_m;  // 64-wide k-blocks of X X^T (ceil(m / 64))
  int nk_n;  // 64-wide k-blocks of A A and B X (ceil(n / 64))
};

// An item: x = kind | group << 2 | flags << 12, y = matrix within group, z = tile row | tile column << 16,
// w = the counter value of the matrix to wait for (0: none).
__host__ __device__ inline int4 ns_item(int kind, int group, int flags, int b, int I, int J, int dep) {
  return make_int4(kind | (group << 2) | (flags << 12), b, I | (J << 16), dep);
}

struct FusedArgs {
  const CUtensorMap* maps;   // [group][kNumRoles], 64-byte aligned
  const NsGroup* groups;
  const int4* items;         // cluster L walks items[begin[L] .. begin[L + 1])
  const int* begin;
  int* counters;             // per matrix (group order): epilogue halves finished in this launch
  unsigned int* done;        // CTAs finished; the last one zeroes the counters and this ticket
  const float* post;         // per matrix: scale folded into the first iteration, or null
  int num_slots;
  int num_groups;
  int c_nonzero;
  float a, b, c;
  int carry;                 // X carried as bf16 hi + lo between combines
  int final_mode;            // 1: the last combine writes the caller's matrices through `fin`
  int* err;
  unsigned long long* clk;
  uint64_t wait_ns;          // limit of every bounded wait (0: kWaitLimitNs); the self-test shortens it
};

template <int kStages>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_fused_kernel(const __grid_constant__ FusedArgs args, const __grid_constant__ FinalArgs<kMaxFinal> fin) {
  using S = GemmShape<true, 256, kStages>;
  constexpr int BM = S::BM, BK = S::BK, kBN = 256;
  constexpr uint32_t A_BYTES = S::A_BYTES, B_BYTES = S::B_BYTES;
  constexpr uint32_t kIdescK = instr_desc_bf16(2 * BM, kBN, false);   // Gram: B operand K-major
  constexpr uint32_t kIdescMN = instr_desc_bf16(2 * BM, kBN, true);   // combine: B operand MN-major
  constexpr uint16_t kPairMask = 0x3;
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
  const int list = blockIdx.x / kCluster;
  const int t_begin = args.begin[list], t_end = args.begin[list + 1];
  const uint64_t lim = args.wait_ns ? args.wait_ns : kWaitLimitNs;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (kStages + st); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
  auto addend_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
  auto map_of = [&](int g, int role) { return args.maps + g * kNumRoles + role; };

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * (kEpilogueThreads / 32));  // every epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(addend_bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    for (int i = lane; i < args.num_groups * kNumRoles; i += 32) tma_prefetch_map(args.maps + i);
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
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      for (int t = t_begin; t < t_end; ++t) {
        const int4 it = __ldg(args.items + t);
        const int kind = it.x & 3, g = (it.x >> 2) & 1023, flags = it.x >> 12;
        const int I = (it.z & 0xFFFF) + rank, J = it.z >> 16;
        const NsGroup G = args.groups[g];
        if (it.w > 0 && !wait_counter_bounded(args.counters + G.first_slot + it.y, it.w, abort_flag, args.err, lim))
          break;
        fence_proxy_async_global();
        const bool gram = kind != kNsComb;
        const bool odd = (flags & kNsOdd) != 0;
        const CUtensorMap *ma, *mb;
        int nk;
        if (kind == kNsGram) {
          ma = mb = map_of(g, odd ? kRoleX1 : kRoleX0);
          nk = G.nk_m;
        } else if (kind == kNsGramAA) {
          ma = mb = map_of(g, kRoleA);
          nk = G.nk_n;
        } else {
          ma = map_of(g, kRoleP);
          mb = map_of(g, odd ? kRoleXmn1 : kRoleXmn0);
          nk = G.nk_n;
        }
        // Gram tiles whose 128 A rows are this CTA's half of the B block read A from B's copy.
        const bool a_in_b = gram && ((I >> 1) == J);
        const uint32_t bytes = a_in_b ? B_BYTES : A_BYTES + B_BYTES;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, args.err, lim)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(full_bar(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * bytes);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (!a_in_b) tma_load_3d_pair(smem_u32(sA + stage * A_BYTES), ma, leader_full, kb * BK, I * BM, it.y);
          const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
          if (gram) {  // this CTA's 128 of the 256 B rows
            tma_load_3d_pair(b_dst, mb, leader_full, kb * BK, J * kBN + rank * 128, it.y);
          } else {     // this CTA's 128 of the 256 B columns, two boxes of 64
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_3d_pair(b_dst + c * 8192u, mb, leader_full, J * kBN + rank * 128 + c * 64, kb * BK, it.y);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag && rank == 0) {
        for (int st = 0; st < kStages; ++st)
          if (armed & (1u << st)) mbar_wait_drain(full_bar(st), (armed_parity >> st) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool issued = false;
      for (int t = t_begin; t < t_end; ++t) {
        const int4 it = __ldg(args.items + t);
        const int kind = it.x & 3, g = (it.x >> 2) & 1023;
        const int I = it.z & 0xFFFF, J = it.z >> 16;  // this CTA's rows (rank 0)
        const bool gram = kind != kNsComb;
        const int nk = kind == kNsGram ? args.groups[g].nk_m : args.groups[g].nk_n;
        const bool a_in_b = gram && ((I >> 1) == J);
        const uint32_t idesc = gram ? kIdescK : kIdescMN;
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err, lim)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.err, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
          const uint32_t a_addr = a_in_b ? b_addr : smem_u32(sA + stage * A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t a_desc = smem_desc_sw128(a_addr + k * 32u, 16u, 1024u);
            const uint64_t b_desc = gram ? smem_desc_sw128(b_addr + k * 32u, 16u, 1024u)
                                         : smem_desc_sw128(b_addr + k * 2048u, 8192u, 1024u);
            mma_bf16_ss_pair(d_tmem, a_desc, b_desc, idesc, (kb | k) != 0 ? 1u : 0u);
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
    // Eight warps, two per TMEM lane quarter; the four warps of a column half share two 128 x 64
    // staging boxes that one thread (the half's leader) moves by TMA. See ns_gemm.cuh.
    constexpr int kHalfCols = kBN / 2;
    constexpr int kBoxes = kHalfCols / 64;
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const bool leader = quarter == 0 && lane == 0;
    const uint32_t half_bar = 1u + static_cast<uint32_t>(half);
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    uint8_t* const stg_base = staging + half * 32768;
    const uint32_t bar_base = addend_bar(2 * half);
    uint32_t box_phase = 0u;
    uint32_t box_pending = 0u;
    auto stg_box = [&](int b) { return stg_base + b * 16384; };
    auto box_bar = [&](int b) { return bar_base + 8u * static_cast<uint32_t>(b); };
    auto sync_half = [&]() { named_barrier_sync(half_bar, 128); };
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
      if (!mbar_wait_bounded(box_bar(b), (box_phase >> b) & 1u, abort_flag, args.err, lim)) return false;
      box_phase ^= 1u << b;
      box_pending &= ~(1u << b);
      return true;
    };
    auto store_box = [&](int b, const CUtensorMap* map, int x, int y, int z) {
      fence_proxy_async_smem();
      sync_half();
      if (leader) {
        tma_store_3d(map, smem_u32(stg_box(b)), x, y, z);
        bulk_commit_group();
      }
    };
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
    int ring = 0;
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
      const int4 it = __ldg(args.items + t);
      const int kind = it.x & 3, g = (it.x >> 2) & 1023, flags = it.x >> 12;
      const int I = (it.z & 0xFFFF) + rank, J = it.z >> 16;
      const int mat = it.y;
      const int slot = args.groups[g].first_slot + mat;
      const bool gram = kind != kNsComb;
      const bool odd = (flags & kNsOdd) != 0;
      const bool has_e = kind != kNsGram;
      const bool carry = !gram && args.carry != 0;
      const bool final_out = !gram && (flags & kNsLast) && args.final_mode;
      // The stage this item's addend comes from has finished once the item's dependency holds.
      if (has_e && it.w > 0 && leader) {
        if (wait_counter_bounded(args.counters + slot, it.w, abort_flag, args.err, lim)) fence_proxy_async_global();
      }
      const CUtensorMap* m_out;
      const CUtensorMap* m_mirror = nullptr;
      const CUtensorMap* m_e = nullptr;
      const CUtensorMap* m_e_lo = nullptr;
      const CUtensorMap* m_out_lo = nullptr;
      float s_acc, s_e = 0.f;
      const float post = ((flags & kNsFirst) && args.post) ? __ldg(args.post + slot) : 1.0f;
      if (kind == kNsGram) {
        const bool to_a = args.c_nonzero != 0;
        m_out = map_of(g, to_a ? kRoleA : kRoleP);
        m_mirror = map_of(g, to_a ? kRoleAm : kRolePm);
        s_acc = (to_a ? 1.0f : args.b) * post * post;
      } else if (kind == kNsGramAA) {
        m_out = map_of(g, kRoleP);
        m_mirror = map_of(g, kRolePm);
        m_e = map_of(g, kRoleA);
        s_acc = args.c;
        s_e = args.b;
      } else {
        m_e = map_of(g, odd ? kRoleX1 : kRoleX0);
        m_out = map_of(g, odd ? kRoleX0 : kRoleX1);
        m_e_lo = map_of(g, odd ? kRoleLo1 : kRoleLo0);
        m_out_lo = map_of(g, odd ? kRoleLo0 : kRoleLo1);
        s_acc = post;
        s_e = args.a * post;
      }
      const int block_col = 2 * J + half;
      const bool skip = gram && (block_col < I);
      const bool mirror = gram && (block_col > I);
      const int col_base = J * kBN + half * kHalfCols;
      const int y_tile = I * BM;
      // Addend boxes (the Gram of X has none): box 0 may reuse its staging box once all but the latest
      // store have read theirs, box 1 once all have; under the precise carry the two boxes hold one
      // unit's high and low parts.
      if (has_e && !skip) {
        if (carry) {
          load_box(0, m_e, col_base, y_tile, mat, true);
          load_box(1, m_e_lo, col_base, y_tile, mat, true);
        } else {
          load_box(0, m_e, col_base, y_tile, mat, false);
          load_box(1, m_e, col_base + 64, y_tile, mat, true);
        }
      }
      mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.err, lim);
      tc_fence_after();
      bool released = false;
      if (carry && !skip) {
#pragma unroll 1
        for (int box = 0; box < kBoxes; ++box) {
          const int x0 = col_base + box * 64;
          if (box == 1) {
            load_box(0, m_e, x0, y_tile, mat, true);
            load_box(1, m_e_lo, x0, y_tile, mat, true);
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
          if (box == kBoxes - 1) {  // the whole accumulator is read: hand it back before the addend wait
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            released = true;
          }
          add_carried_addend(v, s_e);
          uint8_t* rh = stg_box(0) + (quarter * 32 + lane) * 128;
          uint8_t* rl = stg_box(1) + (quarter * 32 + lane) * 128;
          if (final_out) {
            const int mi = slot;
            const bool tr = fin.trans[mi] != 0;
            const float us = fin.scale[mi];
            const int ux = tr ? y_tile : x0, uy = tr ? x0 : y_tile;
            if (fin.update) {
              fence_proxy_async_smem();
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
            store_box(0, m_out, x0, y_tile, mat);
            store_box(1, m_out_lo, x0, y_tile, mat);
          }
        }
      } else if (final_out) {
        // Both boxes of X_k into registers as bf16, the accumulator released at once, then the
        // caller's two boxes loaded in place of the addends: W' = keep * W - scale * X_k, or out = X_k.
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
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
        released = true;
        const int mi = slot;
        const bool tr = fin.trans[mi] != 0;
        const float us = fin.scale[mi];
        if (fin.update) {
          fence_proxy_async_smem();
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
          if (box == kBoxes - 1) {  // the whole accumulator is read: hand it back before the stores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            released = true;
          }
          const int x0 = col_base + box * 64;
          const int b = has_e ? box : (ring & 1);
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
            free_box(false);
            ++ring;
          }
          {
            uint32_t packed[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) packed[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(row_ptr + ((j ^ (lane & 7)) * 16)) =
                  make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
            store_box(b, m_out, x0, y_tile, mat);
            if (mirror) {
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
              store_box(bm, m_mirror, y_tile, x0, mat);
            }
          }
        }
      }
      // Every warp of the half takes the same decision: one that read the flag before another thread
      // raised it would otherwise go on alone and wait at the next named barrier for ever.
      if (named_barrier_or(half_bar, 128, *abort_flag != 0)) break;
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      // This half of the tile is in global memory: count it for the matrix's next stage.
      if (leader) {
        bulk_wait_group0();
        fence_proxy_async_global();
        red_release_gpu_add(args.counters + slot, 1);
      }
    }
    if (leader) {
      for (int b = 0; b < 2; ++b)
        if ((box_pending >> b) & 1u) mbar_wait_drain(box_bar(b), (box_phase >> b) & 1u);
      bulk_wait_group0();
    }
  }

  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's counter updates (ordered before here by the barriers) come first
    if (args.clk) {
      atomicAdd(args.clk, static_cast<unsigned long long>(clock64() - clk_start));
      atomicAdd(args.clk + 1, static_cast<unsigned long long>(global_timer_ns() - ns_start));
    }
    // The last CTA to finish zeroes the counters for the next launch: every other CTA has made its
    // last counter update before its own arrival here.
    if (atom_add_acq_rel_gpu(args.done, 1u) == gridDim.x - 1) {
      for (int i = 0; i < args.num_slots; ++i) args.counters[i] = 0;
      __threadfence();
      *args.done = 0u;
    }
  }
}

}  // namespace muon
