// Pieces shared by the grouped GEMM kernels: the m-tile table built from the
// unit offsets, tile decoding, SiLU, and the timeout report.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kTileRows = 128;   // rows of one m-tile (tokens of one unit)
constexpr int kMaxGroups = 256;

struct Tile {
  int g, row0, rows, nt;
};

// Work item w -> (group, first row, rows, n-tile) for m-tiles of TR rows.
template <int TR = kTileRows>
__device__ __forceinline__ Tile decode_tile(int w, int n_tiles, int n_groups, const int* prefix,
                                            const int* offs) {
  Tile t;
  const int mt = w / n_tiles;
  t.nt = w - mt * n_tiles;
  // largest g in [0, n_groups) with prefix[g] <= mt
  int lo = 0, hi = n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= mt)
      lo = mid;
    else
      hi = mid;
  }
  t.g = lo;
  t.row0 = offs[lo] + (mt - prefix[lo]) * TR;
  t.rows = min(TR, offs[lo + 1] - t.row0);
  return t;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Epilogue staging of one warp's 32 output rows x 64 bf16 columns (4 KB,
// 1024-byte aligned) in the layout a TMA store with the 128-byte swizzle
// reads: 16-byte chunk c of row r sits at chunk c ^ (r % 8) of the row, so
// the eight lanes writing one chunk index hit eight different bank groups.
constexpr uint32_t kStageRowsBytes = 32 * 128;

// Lane `lane` writes chunks c0 .. c0 + 3 (32 columns) of its row.
__device__ __forceinline__ void stage_row_32(uint8_t* buf, int lane, int c0,
                                             const uint32_t (&pk)[16]) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<uint4*>(row + (((c0 + i) ^ (lane & 7)) << 4)) =
        make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

__device__ __forceinline__ void fail(volatile int* abort, int32_t* status) {
  *abort = 1;
  report(status, MOE_ERR_DEVICE_TIMEOUT);
}


// Built by one warp (m-tiles of TR rows): s_prefix[g] = first m-tile of group g (s_prefix[G] =
// total), s_offs = row offsets, *s_total = number of m-tiles.  offsets ==
// nullptr means one dense group of dense_rows rows.  Offsets that decrease,
// are negative, or end past out_rows are reported (MOE_ERR_BAD_INDEX) and
// give zero tiles.
template <int TR = kTileRows>
__device__ __forceinline__ void build_tile_table(const int32_t* offsets, int G, int dense_rows,
                                                 long long out_rows, int* s_prefix, int* s_offs,
                                                 int* s_total, int32_t* status, int lane) {
  if (offsets == nullptr) {
    if (lane == 0) {
      s_offs[0] = 0;
      s_offs[1] = dense_rows;
      s_prefix[0] = 0;
      s_prefix[1] = (dense_rows + TR - 1) / TR;
      *s_total = s_prefix[1];
    }
    return;
  }
  // every offset in flight at once (lane-strided), then per-lane runs from
  // shared memory
  constexpr int kPer = (kMaxGroups + 1 + 31) / 32;
  int ov[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int g = lane + 32 * i;
    ov[i] = g <= G ? offsets[g] : 0;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int g = lane + 32 * i;
    if (g <= G) s_offs[g] = ov[i];
  }
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
      local += b > a ? (b - a + TR - 1) / TR : 0;
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
      const int a = s_offs[g], b = s_offs[g + 1];
      run += b > a ? (b - a + TR - 1) / TR : 0;
    }
  }
  if (lane == 31) {
    const int last = s_offs[G];
    bad |= static_cast<long long>(last) > out_rows;
    s_prefix[G] = incl;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 31) *s_total = bad ? 0 : incl;
  if (bad && lane == 0) report(status, MOE_ERR_BAD_INDEX);
}

}  // namespace moe
