// Grouped GEMM of the expert FFN on CTA pairs: two CTAs of a cluster share
// one tcgen05.mma.cta_group::2 of N = 256 and M = 256 (128 rows per CTA) or
// M = 128 (64 rows per CTA).
//
//   D[r, n] = sum_k A[r, k] * B[b_row(g, n), k]      r in the rows of group g
//
// Why pairs: with one CTA per 128 x 256 tile, each SM stages the whole 256-row
// weight slab of every k-block (48 KB per stage with the token rows).  A pair
// splits the weight slab between the two SMs (each stages 128 rows, 32 KB per
// stage) and the MMA reads each half from the SM that holds it, so the bytes
// that enter each SM drop by a third and six ring stages fit where four did.
//
// Tiles.  Dense GEMMs (one group) use 256-row tiles.  Routed GEMMs split each
// unit of c rows into 256-row tiles plus, when the remainder r = c mod 256 is
// in (0, 128], one 128-row tile (M = 128: 64 rows per CTA), so a unit's last
// tile pads to a multiple of 128 rows, as with single CTAs, while its other
// rows run at the pair's cost.  CTA rank q takes rows [q R, q R + R) of a tile
// (R = 128 or 64).
//
// Accumulator placement (both per CTA): M = 256, lane l holds the CTA's row l
// over all N columns; M = 128, lanes 0-63 hold its rows 0-63 over columns
// [0, N/2) and lanes 64-127 the same rows over [N/2, N), each in N/2 TMEM
// columns.
//
// B staging (what each CTA's half of N holds):
//   EPI_SWIGLU  rank q stages gate rows [64 q, 64 q + 64) then the matching up
//               rows of the item's 128 neurons, so every 128-column half of N
//               is gate(64) | up(64) of 64 neurons and a thread finds both
//               operands of its SiLU(gate) * up in its own lane (MoE-Prism,
//               arXiv 2510.19366, §III-B1 Eq. (1)); 128 outputs per item
//   EPI_BF16    rank q stages output columns [128 q, 128 q + 128) of a 256-wide
//               n-tile (down projection, X' = A Wdown)
//
// Roles:
//   warp 0      TMA producer of this CTA's B half (and its A rows unless the
//               kernel gathers them); every load counts its bytes on the
//               LEADER's (rank 0's) `full` barrier, which the leader's
//               producer alone arms with the bytes of both CTAs
//   warp 1      allocates the pair's TMEM; on the leader one elected thread
//               issues the pair MMAs and commits to both CTAs' `empty` and
//               `tfull` barriers (multicast)
//   warps 2..5  epilogue of this CTA's rows from its own TMEM; releases the
//               accumulator on the leader's `tempty` (8 arrivals); full 32-row
//               slabs leave through TMA stores, partial ones through masked
//               16-byte stores
//   GATHER: warps 6..9 copy this CTA's token rows of every k-block straight
//               from x (row r = token gtok[row]) with cp.async into the
//               swizzled A stage.  Rank 0's copies arrive on the leader's
//               `full` directly; rank 1's arrive on its local `afull`, and
//               warp 10 of rank 1 forwards each completed stage to the
//               leader's `full` with one cluster-scope release (a release
//               costs ~300 cycles, and ~1000 in a thread with copies still in
//               flight, so it is paid once per stage by a thread that has
//               none)
// Every wait is bounded (MOE_ERR_DEVICE_TIMEOUT).  Both CTAs meet at a cluster
// barrier after set-up (no remote arrive before the barriers exist) and
// before TMEM is freed and the CTAs exit (no MMA or arrive still aimed at a
// CTA that has gone).
#include <cudaTypedefs.h>

#include "gemm_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BM = kTileRows;   // token rows per CTA of a 256-row tile
constexpr int BK = 64;
constexpr int BN = 256;         // N of one pair MMA
constexpr int kBaseThreads = 192;
constexpr int kGatherThreads = 128;                          // warps 6..9
constexpr int kGatherKernelThreads = kBaseThreads + kGatherThreads + 32;  // + relay warp 10
constexpr uint32_t kABytes = BM * BK * 2;
constexpr uint32_t kBBytes = (BN / 2) * BK * 2;
constexpr uint32_t kTmemCols = 2 * BN;

template <int STAGES>
struct PairCfg {
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = STAGES * kABytes;
  static constexpr uint32_t kOffStage = STAGES * (kABytes + kBBytes);  // 4 epilogue buffers
  static constexpr uint32_t kOffBar = kOffStage + 4 * kStageRowsBytes;
  static constexpr uint32_t kNumBars = 3 * STAGES + 5;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffPrefix = kOffMisc + 16;
  static constexpr uint32_t kOffOffs = kOffPrefix + (kMaxGroups + 1) * 4;
  static constexpr uint32_t kSmemUsed = kOffOffs + (kMaxGroups + 1) * 4;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct PairParams {
  const int32_t* offsets;
  int n_groups;
  int dense_rows;
  int K;
  int n_tiles;        // n-tiles per group
  int bn_out;         // output columns per n-tile
  int b_group_rows;   // rows of B per group
  int b_up_offset;    // SWIGLU: rows between a gate row and its up row
  int tails;          // routed: a unit's remainder of <= 128 rows is one M = 128 tile
  const uint4* gx;    // GATHER: A rows are x[gtok[r]] (bf16 [*, K]), 16-byte vectors
  const int32_t* gtok;
  int gx_rows;
  void* out;
  long long ld_out;
  long long out_rows;
  int32_t* status;
  uint32_t debug_flags;
};

struct PTile {
  int g, row0, rows, nt;
  bool m128;   // M = 128 tile (64 rows per CTA)
};

// 256-row and 128-row tiles of a unit of c rows.
__device__ __forceinline__ void unit_tiles(int c, int tails, int& n256, int& n128) {
  if (c <= 0) {
    n256 = n128 = 0;
    return;
  }
  const int r = c & 255;
  if (!tails) {
    n256 = (c + 255) >> 8;
    n128 = 0;
  } else {
    n256 = (c >> 8) + (r > 128 ? 1 : 0);
    n128 = (r > 0 && r <= 128) ? 1 : 0;
  }
}

// Built by one warp: s_prefix[g] = first tile of group g, s_offs = offsets,
// *s_total = tiles.  Offsets that decrease, are negative, or end past
// out_rows are reported and give zero tiles.
__device__ __forceinline__ void build_pair_table(const int32_t* offsets, int G, int dense_rows,
                                                 long long out_rows, int tails, int* s_prefix,
                                                 int* s_offs, int* s_total, int32_t* status,
                                                 int lane) {
  if (offsets == nullptr) {
    if (lane == 0) {
      s_offs[0] = 0;
      s_offs[1] = dense_rows;
      s_prefix[0] = 0;
      s_prefix[1] = (dense_rows + 255) / 256;
      *s_total = s_prefix[1];
    }
    return;
  }
  for (int g = lane; g <= G; g += 32) s_offs[g] = offsets[g];
  __syncwarp();
  const int per = (G + 31) / 32;
  const int g0 = lane * per;
  int local = 0;
  bool bad = false;
  for (int i = 0; i < per; ++i) {
    const int g = g0 + i;
    if (g < G) {
      const int a = s_offs[g], b = s_offs[g + 1];
      bad |= (a < 0) || (b < a);
      int n256, n128;
      unit_tiles(b - a, tails, n256, n128);
      local += n256 + n128;
    }
  }
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - local;
  for (int i = 0; i < per; ++i) {
    const int g = g0 + i;
    if (g < G) {
      s_prefix[g] = run;
      int n256, n128;
      unit_tiles(s_offs[g + 1] - s_offs[g], tails, n256, n128);
      run += n256 + n128;
    }
  }
  if (lane == 31) {
    bad |= static_cast<long long>(s_offs[G]) > out_rows;
    s_prefix[G] = incl;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 31) *s_total = bad ? 0 : incl;
  if (bad && lane == 0) report(status, MOE_ERR_BAD_INDEX);
}

__device__ __forceinline__ PTile decode_pair_tile(int w, int n_tiles, int n_groups, int tails,
                                                  const int* prefix, const int* offs) {
  PTile t;
  const int mt = w / n_tiles;
  t.nt = w - mt * n_tiles;
  int lo = 0, hi = n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= mt)
      lo = mid;
    else
      hi = mid;
  }
  t.g = lo;
  const int a = offs[lo], c = offs[lo + 1] - a;
  int n256, n128;
  unit_tiles(c, tails, n256, n128);
  const int i = mt - prefix[lo];
  t.m128 = i >= n256;
  t.row0 = a + (t.m128 ? 256 * n256 : 256 * i);
  t.rows = min(t.m128 ? 128 : 256, a + c - t.row0);
  return t;
}

// Bounded wait with cluster-scope acquire: pairs with a remote release
// arrive (the relay of rank 1's gathered rows).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void mbar_arrive_remote_release_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

template <int EPI, int STAGES, bool GATHER>
__global__ void __launch_bounds__(GATHER ? kGatherKernelThreads : kBaseThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmA64,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmOut, const PairParams p) {
  using C = PairCfg<STAGES>;
  extern __shared__ uint8_t smem_raw[];
  // The dynamic shared window starts at the same offset in both CTAs, so the
  // aligned base (and every barrier and stage) sits at the same offset too.
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;                 // leader only
  uint64_t* empty = bars + STAGES;
  uint64_t* afull = bars + 2 * STAGES;   // rank 1, GATHER only
  uint64_t* tfull = bars + 3 * STAGES;
  uint64_t* tempty = tfull + 2;          // leader only
  uint64_t* done = tempty + 2;           // leader only
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int* s_total = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  int* s_prefix = reinterpret_cast<int*>(smem + C::kOffPrefix);
  int* s_offs = reinterpret_cast<int*>(smem + C::kOffOffs);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // set-up that reads nothing written upstream runs before the grid
  // dependency wait, overlapping the previous kernel's tail
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // GATHER: the producer's arrive (B bytes), rank 0's gather threads and
      // the relay of rank 1's stage
      mbar_init(&full[s], GATHER ? 1 + kGatherThreads + 1 : 1);
      mbar_init(&empty[s], 1);
      mbar_init(&afull[s], kGatherThreads);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 8);
    mbar_init(&tempty[1], 8);
    mbar_init(done, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA64);
    }
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  pdl_wait_and_trigger();
  if (warp == 2)
    build_pair_table(p.offsets, p.n_groups, p.dense_rows, p.out_rows, p.tails, s_prefix, s_offs,
                     s_total, p.status, lane);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total_work = *s_total * p.n_tiles;
  const int KB = p.K / BK;
  const int G = p.offsets == nullptr ? 1 : p.n_groups;
  const int tails = p.offsets == nullptr ? 0 : p.tails;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full_l = mapa_shared(smem_u32(full), 0);  // leader's full[0]
      int stage = 0;
      uint32_t phase = 0;
      bool skip = leader && (p.debug_flags & MOE_DEBUG_SKIP_FIRST_LOAD) != 0u;
      bool ok = true;
      for (int w = cid; ok && w < total_work; w += ncl) {
        const PTile t = decode_pair_tile(w, p.n_tiles, G, tails, s_prefix, s_offs);
        const int R = t.m128 ? BM / 2 : BM;
        const int row0 = t.row0 + static_cast<int>(rank) * R;
        const uint32_t a_bytes = GATHER ? 0u : static_cast<uint32_t>(R) * BK * 2;
        const int b_row = EPI == EPI_SWIGLU
                              ? t.g * p.b_group_rows + t.nt * p.bn_out + static_cast<int>(rank) * 64
                              : t.g * p.b_group_rows + t.nt * p.bn_out +
                                    static_cast<int>(rank) * (BN / 2);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: the MMA's wait on this slot must time out
          } else {
            const uint32_t fb = full_l + 8u * static_cast<uint32_t>(stage);
            uint8_t* sa = smem + C::kOffA + stage * kABytes;
            uint8_t* sb = smem + C::kOffB + stage * kBBytes;
            if (leader) mbar_expect_tx(&full[stage], 2 * (kBBytes + a_bytes));
            if (!GATHER) tma_load_2d_pair(sa, t.m128 ? &tmA64 : &tmA, fb, kb * BK, row0);
            if (EPI == EPI_SWIGLU) {
              tma_load_2d_pair(sb, &tmB, fb, kb * BK, b_row);
              tma_load_2d_pair(sb + 64 * BK * 2, &tmB, fb, kb * BK, b_row + p.b_up_offset);
            } else {
              tma_load_2d_pair(sb, &tmB, fb, kb * BK, b_row);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        fail(s_abort, p.status);
      } else {
        // Wait for the MMA's release of every slot: its last commits arrive
        // on this CTA's `empty` barriers and must not outlive the CTA.  The
        // same wait covers this CTA's loads (each was consumed by an MMA).
        for (int i = 0; i < STAGES; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, nullptr)) {
            fail(s_abort, p.status);
            break;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader && lane == 0) {
      constexpr uint32_t idesc256 = idesc_bf16_f32(2 * BM, BN);
      constexpr uint32_t idesc128 = idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int w = cid; ok && w < total_work; w += ncl) {
        const PTile t = decode_pair_tile(w, p.n_tiles, G, tails, s_prefix, s_offs);
        const uint32_t idesc = t.m128 ? idesc128 : idesc256;
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          const bool got = GATHER ? mbar_wait_cluster(&full[stage], phase, s_abort)
                                  : mbar_wait(&full[stage], phase, s_abort);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(smem + C::kOffA + stage * kABytes));
          const uint64_t bd = sdesc_sw128(smem_u32(smem + C::kOffB + stage * kBBytes));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16_pair(d, ad + 2u * k, bd + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(&empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) fail(s_abort, p.status);
      // every MMA issued here must be complete before either CTA frees TMEM
      umma_commit_pair(done, 0x1);
      mbar_wait(done, 0u, nullptr);
    }
    __syncwarp();
  } else if (warp < 6) {
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t tempty_l = mapa_shared(smem_u32(tempty), 0);  // leader's tempty[0]
    uint8_t* sbuf = smem + C::kOffStage + q * kStageRowsBytes;
    int acc = 0;
    uint32_t aphase = 0;
    for (int w = cid; w < total_work; w += ncl) {
      const PTile t = decode_pair_tile(w, p.n_tiles, G, tails, s_prefix, s_offs);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], aphase, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) fail(s_abort, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // rows of this warp's slab within the tile, and the part of N it holds
      const int R = t.m128 ? BM / 2 : BM;
      const int slab0 = static_cast<int>(rank) * R + (t.m128 ? (q & 1) * 32 : q * 32);
      const int nhalf = t.m128 ? (q >> 1) : 0;   // M = 128: lanes 64-127 hold N/2..N
      const int r_tile = slab0 + lane;
      const long long grow = static_cast<long long>(t.row0) + r_tile;
      const bool valid = r_tile < t.rows && grow < p.out_rows;
      const bool full_slab =
          slab0 + 32 <= t.rows && static_cast<long long>(t.row0) + slab0 + 32 <= p.out_rows;
      // 32-column chunks: TMEM column of the value (SWIGLU: the gate; its up
      // value sits 64 columns on) and the output column within the n-tile
      const int n_chunks = EPI == EPI_SWIGLU ? (t.m128 ? 2 : 4) : (t.m128 ? 4 : 8);
      const int col_base = t.nt * p.bn_out + nhalf * (EPI == EPI_SWIGLU ? 64 : BN / 2);
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out + col_base;
#pragma unroll 1
      for (int ci = 0; ci < n_chunks; ++ci) {
        uint32_t pk[16];
        int ocol;   // output column of this chunk, from col_base
        if (EPI == EPI_SWIGLU) {
          // chunk ci: gate at TMEM column (ci / 2) * 128 + (ci % 2) * 32,
          // up 64 columns further; outputs 32 ci .. 32 ci + 31
          const int tc = (ci >> 1) * 128 + (ci & 1) * 32;
          ocol = ci * 32;
          uint32_t gv[32], uv[32];
          tmem_ld32(tbase + tc, gv);
          tmem_ld32(tbase + tc + 64, uv);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = silu_f(__uint_as_float(gv[2 * i])) * __uint_as_float(uv[2 * i]);
            const float a1 =
                silu_f(__uint_as_float(gv[2 * i + 1])) * __uint_as_float(uv[2 * i + 1]);
            pk[i] = pack_bf16x2(a0, a1);
          }
        } else {
          ocol = ci * 32;
          uint32_t v[32];
          tmem_ld32(tbase + ci * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        }
        if (full_slab) {
          if ((ci & 1) == 0) {  // first half of a 64-column block: buffer free?
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          stage_row_32(sbuf, lane, (ci & 1) * 4, pk);
          if ((ci & 1) != 0) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, sbuf, col_base + ocol - 32, t.row0 + slab0);
              bulk_commit();
            }
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ocol);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_l + 8u * static_cast<uint32_t>(acc));
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();  // stores done before the CTA (and its smem) goes
    __syncwarp();
  } else if (GATHER && warp < 10) {
    // Row gather: thread g copies 16-byte chunk (g % 8) of rows g / 8 + 16 i
    // of every k-block; the chunk lands at chunk ^ (row % 8) of its 128-byte
    // row (the 128-byte swizzle the MMA descriptors expect).  The copies of a
    // stage are one cp.async group; once a group is LAG groups old the thread
    // waits for it, orders it for the tensor cores' async-proxy reads and
    // arrives (rank 0: the leader's `full`; rank 1: its `afull`, which the
    // relay forwards).
    constexpr int LAG = STAGES - 2;
    const int g = threadIdx.x - kBaseThreads;
    const int chunk = g & 7, rg = g >> 3;
    const uint32_t dst_off = static_cast<uint32_t>(rg * 128 + ((chunk ^ (rg & 7)) << 4));
    const size_t nv = static_cast<size_t>(p.K) / 8;
    uint64_t* arrive_bar = leader ? full : afull;
    int stage = 0, astage = 0, pending = 0;
    uint32_t phase = 0;
    bool ok = true, bad = false;
    for (int w = cid; ok && w < total_work; w += ncl) {
      const PTile t = decode_pair_tile(w, p.n_tiles, G, tails, s_prefix, s_offs);
      const int R = t.m128 ? BM / 2 : BM;
      const int base = t.row0 + static_cast<int>(rank) * R;
      const int n_valid = min(max(t.rows - static_cast<int>(rank) * R, 0), R);
      const uint4* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rg + 16 * i;
        int tok = -1;
        if (r < n_valid) {
          tok = __ldg(p.gtok + base + r);
          if (tok < 0 || tok >= p.gx_rows) {
            bad = true;
            tok = -1;
          }
        }
        src[i] = tok >= 0 ? p.gx + static_cast<size_t>(tok) * nv + chunk : nullptr;
      }
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + C::kOffA + stage * kABytes) + dst_off;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (src[i] != nullptr)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa + i * 16 * 128),
                         "l"(src[i] + kb * (BK / 8))
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (++pending > LAG) {
          asm volatile("cp.async.wait_group %0;" ::"n"(LAG) : "memory");
          fence_proxy_async_smem();
          mbar_arrive(&arrive_bar[astage]);
          if (++astage == STAGES) astage = 0;
          --pending;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (ok) {
      fence_proxy_async_smem();
      for (; pending > 0; --pending) {
        mbar_arrive(&arrive_bar[astage]);
        if (++astage == STAGES) astage = 0;
      }
    } else {
      fail(s_abort, p.status);
    }
    if (bad) report(p.status, MOE_ERR_BAD_INDEX);
  } else if (GATHER && warp == 10) {
    // Relay (rank 1): every stage its gather threads completed is forwarded
    // to the leader's `full` with one cluster-scope release arrive.
    if (!leader && lane == 0) {
      const uint32_t full_l = mapa_shared(smem_u32(full), 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = cid; ok && w < total_work; w += ncl) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&afull[stage], phase, s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_remote_release_cluster(full_l + 8u * static_cast<uint32_t>(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) fail(s_abort, p.status);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

template <typename K>
cudaError_t max_pair_clusters(K kern, int threads, int smem, int sm_count, int* out) {
  static int cached[64][2] = {{0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int slot = threads == kBaseThreads ? 0 : 1;
  if (cached[dev][slot] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count / 2));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    cached[dev][slot] = n > 0 ? n : 1;
  }
  *out = cached[dev][slot];
  return cudaSuccess;
}

template <int EPI, int STAGES, bool GATHER>
cudaError_t run_pair(const GemmArgs& g, cudaStream_t s) {
  using C = PairCfg<STAGES>;
  CUtensorMap ta, ta64, tb, to;
  if (GATHER) {
    if (g.gather_x == nullptr || g.gather_tok == nullptr) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&ta, g.gather_x, 1, g.K, 1)) return cudaErrorInvalidValue;  // unused
    ta64 = ta;
  } else {
    if (!make_tmap_bf16(&ta, g.a, g.a_rows, g.K, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&ta64, g.a, g.a_rows, g.K, BM / 2)) return cudaErrorInvalidValue;
  }
  if (!make_tmap_bf16(&tb, g.b, g.b_rows, g.K, EPI == EPI_SWIGLU ? 64 : BN / 2))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&to, g.out, g.out_rows, static_cast<int>(g.ld_out), 32))
    return cudaErrorInvalidValue;
  PairParams kp;
  kp.offsets = g.offsets;
  kp.n_groups = g.offsets == nullptr ? 1 : g.n_groups;
  kp.dense_rows = g.dense_rows;
  kp.K = g.K;
  kp.bn_out = EPI == EPI_SWIGLU ? BN / 2 : BN;
  kp.n_tiles = g.n_out / kp.bn_out;
  kp.b_group_rows = g.b_group_rows;
  kp.b_up_offset = EPI == EPI_SWIGLU ? g.n_out : 0;
  kp.tails = g.offsets != nullptr ? 1 : 0;
  kp.gx = static_cast<const uint4*>(g.gather_x);
  kp.gtok = g.gather_tok;
  kp.gx_rows = g.gather_rows;
  kp.out = g.out;
  kp.ld_out = g.ld_out;
  kp.out_rows = g.out_rows;
  kp.status = g.status;
  kp.debug_flags = g.debug_flags;
  long long pair_tiles;
  if (g.offsets == nullptr)
    pair_tiles = (g.dense_rows + 2 * BM - 1) / (2 * BM);
  else
    pair_tiles = (g.max_rows_hint + 2 * BM - 1) / (2 * BM) + 2 * g.n_groups;
  const long long work = pair_tiles * kp.n_tiles;
  if (work <= 0) return cudaSuccess;
  auto kern = grouped_gemm_pair_kernel<EPI, STAGES, GATHER>;
  constexpr int threads = GATHER ? kGatherKernelThreads : kBaseThreads;
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(kern, static_cast<int>(C::kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  int max_cl = 1;
  e = max_pair_clusters(kern, threads, static_cast<int>(C::kSmemBytes), g.sm_count, &max_cl);
  if (e != cudaSuccess) return e;
  const int clusters = static_cast<int>(work < max_cl ? work : max_cl);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ta, ta64, tb, to, kp);
}

}  // namespace

bool gemm_pair_supports(int epi, int n_out) {
  if (epi == EPI_SWIGLU) return n_out % (BN / 2) == 0;
  if (epi == EPI_BF16) return n_out % BN == 0;
  return false;
}

cudaError_t launch_gemm_pair(const GemmArgs& g, cudaStream_t s) {
  if (!gemm_pair_supports(g.epi, g.n_out)) return cudaErrorInvalidValue;
  if (g.epi == EPI_SWIGLU) {
    if (g.gather_x != nullptr) return run_pair<EPI_SWIGLU, 6, true>(g, s);
    return run_pair<EPI_SWIGLU, 6, false>(g, s);
  }
  return run_pair<EPI_BF16, 6, false>(g, s);
}

}  // namespace moe
