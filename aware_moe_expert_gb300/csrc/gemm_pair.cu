// Grouped GEMM of the expert FFN on CTA pairs: two CTAs of a cluster share
// one tcgen05.mma.cta_group::2 of M = 256 (128 token rows each), N = 256.
//
//   D[r, n] = sum_k A[r, k] * B[b_row(g, n), k]      r in the rows of group g
//
// Why pairs: with one CTA per 128 x 256 tile, each SM stages the whole 256-row
// weight slab of every k-block (48 KB per stage with the token rows) and its
// tensor core reads 12 KB of shared memory per 128-cycle MMA.  A pair splits
// the weight slab between the two SMs (each stages 128 rows, 32 KB per stage)
// and the MMA reads each half from the SM that holds it, so weight traffic
// from L2 into the SMs and shared-memory reads per SM both drop by a third,
// and six ring stages fit where four did.
//
// Work items are (pair tile, n-tile): a pair tile is 256 consecutive rows of
// one group (unit), of which CTA rank r takes rows 128 r .. 128 r + 127; the
// last pair tile of a group may leave rank 1 with no valid rows (its loads
// read past the group and its stores are dropped).
//   EPI_SWIGLU  rank 0 stages the gate slab of 128 neurons, rank 1 the matching
//               up slab, so each CTA's accumulator row holds gate | up of its
//               token: act = SiLU(gate) * up, 128 outputs per item
//               (MoE-Prism, arXiv 2510.19366, §III-B1 Eq. (1))
//   EPI_BF16    rank r stages output rows 128 r .. 128 r + 127 of a 256-wide
//               n-tile (down projection, X' = A Wdown)
//
// Roles (both CTAs run all of them unless noted):
//   warp 0      TMA producer of this CTA's half of each stage; every load
//               counts its bytes on the LEADER's (rank 0's) `full` barrier,
//               which the leader's producer alone arms with the bytes of
//               both halves (a remote arm would need a cluster-scope release,
//               a fence per stage that stalls the producer)
//   warp 1      allocates the pair's TMEM; on the leader one elected thread
//               issues the pair MMAs and commits to both CTAs' `empty` and
//               `tfull` barriers (multicast)
//   warps 2..5  epilogue of this CTA's 128 rows from its own TMEM; releases
//               the accumulator on the leader's `tempty` (8 arrivals).  A
//               warp whose 32 rows all belong to the item's unit stages each
//               32 x 64 block of results in shared memory and writes it with
//               one TMA store (full 128-byte lines, off the load/store
//               pipe); the last, partial slab of a unit uses masked stores
// Every wait is bounded (MOE_ERR_DEVICE_TIMEOUT).  Both CTAs meet at a cluster
// barrier after set-up (no remote arrive before the barriers exist) and
// before TMEM is freed and the CTAs exit (no MMA or arrive still aimed at a
// CTA that has gone).
#include <cudaTypedefs.h>

#include "gemm_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BM = kTileRows;   // token rows per CTA
constexpr int BK = 64;
constexpr int BN = 256;         // N of one pair MMA
constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;
constexpr uint32_t kBBytes = (BN / 2) * BK * 2;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 2 * BN;

template <int STAGES>
struct PairCfg {
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = STAGES * kABytes;
  static constexpr uint32_t kOffStage = STAGES * kStageBytes;  // 4 epilogue buffers
  static constexpr uint32_t kOffBar = kOffStage + 4 * kStageRowsBytes;
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
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
  int b_half_offset;  // rows of B between rank 0's and rank 1's slab
  void* out;
  long long ld_out;
  long long out_rows;
  int32_t* status;
  uint32_t debug_flags;
};

template <int EPI, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
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
  uint64_t* tfull = bars + 2 * STAGES;
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
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  pdl_wait_and_trigger();
  if (warp == 2)
    build_tile_table<2 * BM>(p.offsets, p.n_groups, p.dense_rows, p.out_rows, s_prefix, s_offs,
                             s_total, p.status, lane);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total_work = *s_total * p.n_tiles;
  const int KB = p.K / BK;
  const int G = p.offsets == nullptr ? 1 : p.n_groups;
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
        const Tile t = decode_tile<2 * BM>(w, p.n_tiles, G, s_prefix, s_offs);
        const int row0 = t.row0 + static_cast<int>(rank) * BM;
        const int b_row = t.g * p.b_group_rows + t.nt * p.bn_out +
                          static_cast<int>(rank) * p.b_half_offset;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: the MMA's wait on this slot must time out
          } else {
            const uint32_t fb = full_l + 8u * static_cast<uint32_t>(stage);
            if (leader) mbar_expect_tx(&full[stage], 2 * kStageBytes);
            tma_load_2d_pair(smem + C::kOffA + stage * kABytes, &tmA, fb, kb * BK, row0);
            tma_load_2d_pair(smem + C::kOffB + stage * kBBytes, &tmB, fb, kb * BK, b_row);
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
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int w = cid; ok && w < total_work; w += ncl) {
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, s_abort)) {
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
  } else {
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in = q * 32 + lane;
    const uint32_t tempty_l = mapa_shared(smem_u32(tempty), 0);  // leader's tempty[0]
    uint8_t* sbuf = smem + C::kOffStage + q * kStageRowsBytes;
    int acc = 0;
    uint32_t aphase = 0;
    for (int w = cid; w < total_work; w += ncl) {
      const Tile t = decode_tile<2 * BM>(w, p.n_tiles, G, s_prefix, s_offs);
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
      const int r_tile = static_cast<int>(rank) * BM + r_in;  // row within the pair tile
      const long long grow = static_cast<long long>(t.row0) + r_tile;
      const bool valid = r_tile < t.rows && grow < p.out_rows;
      // every row of this warp's slab belongs to the item's unit
      const int slab0 = static_cast<int>(rank) * BM + q * 32;
      const bool full_slab =
          slab0 + 32 <= t.rows && static_cast<long long>(t.row0) + slab0 + 32 <= p.out_rows;
      const int col0 = t.nt * p.bn_out;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out + col0;
      constexpr int kCols = EPI == EPI_SWIGLU ? BN / 2 : BN;  // outputs per row
#pragma unroll 1
      for (int c = 0; c < kCols; c += 32) {
        uint32_t pk[16];
        if (EPI == EPI_SWIGLU) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tbase + c, gv);
          tmem_ld32(tbase + BN / 2 + c, uv);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = silu_f(__uint_as_float(gv[2 * i])) * __uint_as_float(uv[2 * i]);
            const float a1 =
                silu_f(__uint_as_float(gv[2 * i + 1])) * __uint_as_float(uv[2 * i + 1]);
            pk[i] = pack_bf16x2(a0, a1);
          }
        } else {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        }
        if (full_slab) {
          if ((c & 32) == 0) {  // first half of a 64-column block: buffer free?
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          stage_row_32(sbuf, lane, (c & 32) >> 3, pk);
          if ((c & 32) != 0) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, sbuf, col0 + c - 32, t.row0 + slab0);
              bulk_commit();
            }
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
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
cudaError_t max_pair_clusters(K kern, int smem, int sm_count, int* out) {
  static int cached[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count / 2));
    cfg.blockDim = dim3(kThreads);
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
    cached[dev] = n > 0 ? n : 1;
  }
  *out = cached[dev];
  return cudaSuccess;
}

template <int EPI, int STAGES>
cudaError_t run_pair(const GemmArgs& g, cudaStream_t s) {
  using C = PairCfg<STAGES>;
  CUtensorMap ta, tb, to;
  if (!make_tmap_bf16(&ta, g.a, g.a_rows, g.K, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, g.b, g.b_rows, g.K, BN / 2)) return cudaErrorInvalidValue;
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
  kp.b_half_offset = EPI == EPI_SWIGLU ? g.n_out : BN / 2;
  kp.out = g.out;
  kp.ld_out = g.ld_out;
  kp.out_rows = g.out_rows;
  kp.status = g.status;
  kp.debug_flags = g.debug_flags;
  long long pair_tiles;
  if (g.offsets == nullptr)
    pair_tiles = (g.dense_rows + 2 * BM - 1) / (2 * BM);
  else
    pair_tiles = (g.max_rows_hint + 2 * BM - 1) / (2 * BM) + g.n_groups;
  const long long work = pair_tiles * kp.n_tiles;
  if (work <= 0) return cudaSuccess;
  auto kern = grouped_gemm_pair_kernel<EPI, STAGES>;
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(kern, static_cast<int>(C::kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  int max_cl = 1;
  e = max_pair_clusters(kern, static_cast<int>(C::kSmemBytes), g.sm_count, &max_cl);
  if (e != cudaSuccess) return e;
  const int clusters = static_cast<int>(work < max_cl ? work : max_cl);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kThreads);
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
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, to, kp);
}

}  // namespace

bool gemm_pair_supports(int epi, int n_out) {
  if (epi == EPI_SWIGLU) return n_out % (BN / 2) == 0;
  if (epi == EPI_BF16) return n_out % BN == 0;
  return false;
}

cudaError_t launch_gemm_pair(const GemmArgs& g, cudaStream_t s) {
  if (!gemm_pair_supports(g.epi, g.n_out)) return cudaErrorInvalidValue;
  if (g.epi == EPI_SWIGLU) return run_pair<EPI_SWIGLU, 6>(g, s);
  return run_pair<EPI_BF16, 6>(g, s);
}

}  // namespace moe
