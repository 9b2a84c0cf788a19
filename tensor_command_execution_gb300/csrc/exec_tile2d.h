// exec_tile2d.h - launch parameters and geometry of the tile2d executor,
// shared by its per-tier device objects (exec_tile2d.cu) and the host code
// that encodes the TMA descriptors (exec_host.cpp).
#pragma once

#include <cuda.h>

#include "cmd_internal.h"

namespace cmdx {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 4;
constexpr int kBarrierBytes = 1024;   // barriers; stages start 1024-byte aligned
constexpr int kBoxBytes = 8192;       // one 64-row box of 128-byte rows


struct Tile2dParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap maps[kMaxLoads];
  void* out[kMaxStores];
  int64_t out_ld[kMaxStores];
  int64_t out_bst[kMaxStores][2];
  uint32_t scal[kMaxScalars];
  uint32_t* err;
  int64_t rows, cols;
  uint64_t timeout_ns;
  uint32_t tiles_r, tiles_c, nb1, n_tiles;
  uint32_t group_rows;  // plain 2-D launches: tile rows walked together (>= 1)
  uint32_t prog, n_loads, n_stages, stage_bytes, tx_bytes, debug;
  uint32_t load_off[kMaxLoads];  // byte offset of load j in a stage
  uint8_t in_dt[kMaxLoads];
  uint8_t in_trans[kMaxLoads];
  uint8_t in_bcast[kMaxLoads];   // the load's other tile dim has stride 0: a one-row box
  uint8_t in_rank[kMaxLoads];    // dims of its TMA descriptor
  uint8_t in_split[kMaxLoads];   // transposed load with its column dim split in (column / 8, column % 8)
  // coordinate of descriptor dims 1..4: 0 the other tile dim, 1 batch b0,
  // 2 batch b1, 3 column / 8, 4 column % 8 (of a split column dim)
  uint8_t in_src[kMaxLoads][4];
};

// Entry points of the objects built from exec_tile2d.cu, one per tier t
// (0..2), view variant x (0 for plain 2-D views, 1 for batch dims, broadcast
// loads or descriptors of rank other than 2) and division variant v.
#define CMDX_DECL_TILE(t, x, v)                                                         \
  cudaError_t tile2d_upload_t##t##n##x##e##v(int slot, const uint32_t* words, int n_words); \
  cudaError_t tile2d_launch_t##t##n##x##e##v(const Tile2dParams& p, cudaStream_t stream);
CMDX_DECL_TILE(0, 0, 0) CMDX_DECL_TILE(0, 1, 0) CMDX_DECL_TILE(1, 0, 0)
CMDX_DECL_TILE(1, 1, 0) CMDX_DECL_TILE(2, 0, 0) CMDX_DECL_TILE(2, 1, 0)
CMDX_DECL_TILE(0, 0, 1) CMDX_DECL_TILE(0, 1, 1) CMDX_DECL_TILE(1, 0, 1)
CMDX_DECL_TILE(1, 1, 1) CMDX_DECL_TILE(2, 0, 1) CMDX_DECL_TILE(2, 1, 1)
#undef CMDX_DECL_TILE

}  // namespace cmdx
