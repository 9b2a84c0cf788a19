// exec_host.cpp - host side of the executors: the tier dispatch of program
// uploads and launches, and the TMA descriptors of the tile2d executor.
#include <cudaTypedefs.h>

#include <cstring>
#include <utility>

#include "exec_tile2d.h"

namespace cmdx {

// the base 4-slot tier's 16-element build serves programs whose loads are all 2-byte
static bool half16(int tier, bool ext, bool half2) { return half2 && tier == kTier4 && !ext; }

int contig_chunk(int tier, bool ext, bool half2) { return 32 * (half16(tier, ext, half2) ? 16 : tier_vec(tier, ext)); }

namespace {

using Upload = cudaError_t (*)(int, const uint32_t*, int);
using ContigLaunch = cudaError_t (*)(const ContigParams&, cudaStream_t);
using GenericLaunch = cudaError_t (*)(const GenericParams&, cudaStream_t);
using TileLaunch = cudaError_t (*)(const Tile2dParams&, cudaStream_t);

// [op-set variant][tier]
constexpr Upload kContigUpload[2][kNumTiers] = {
    {contig_upload_t0e0, contig_upload_t1e0, contig_upload_t2e0, contig_upload_t3e0, contig_upload_t4e0},
    {contig_upload_t0e1, contig_upload_t1e1, contig_upload_t2e1, contig_upload_t3e1, contig_upload_t4e1}};
constexpr Upload kGenericUpload[2][kNumTiers] = {
    {generic_upload_t0e0, generic_upload_t1e0, generic_upload_t2e0, generic_upload_t3e0, generic_upload_t4e0},
    {generic_upload_t0e1, generic_upload_t1e1, generic_upload_t2e1, generic_upload_t3e1, generic_upload_t4e1}};
constexpr ContigLaunch kContigLaunch[2][kNumTiers] = {
    {contig_launch_t0e0, contig_launch_t1e0, contig_launch_t2e0, contig_launch_t3e0, contig_launch_t4e0},
    {contig_launch_t0e1, contig_launch_t1e1, contig_launch_t2e1, contig_launch_t3e1, contig_launch_t4e1}};
constexpr GenericLaunch kGenericLaunch[2][kNumTiers] = {
    {generic_launch_t0e0, generic_launch_t1e0, generic_launch_t2e0, generic_launch_t3e0, generic_launch_t4e0},
    {generic_launch_t0e1, generic_launch_t1e1, generic_launch_t2e1, generic_launch_t3e1, generic_launch_t4e1}};
// [op-set variant][view variant][tier]; the wide tiers have no tile kernel
constexpr Upload kTileUpload[2][2][3] = {
    {{tile2d_upload_t0n0e0, tile2d_upload_t1n0e0, tile2d_upload_t2n0e0},
     {tile2d_upload_t0n1e0, tile2d_upload_t1n1e0, tile2d_upload_t2n1e0}},
    {{tile2d_upload_t0n0e1, tile2d_upload_t1n0e1, tile2d_upload_t2n0e1},
     {tile2d_upload_t0n1e1, tile2d_upload_t1n1e1, tile2d_upload_t2n1e1}}};
constexpr TileLaunch kTileLaunch[2][2][3] = {
    {{tile2d_launch_t0n0e0, tile2d_launch_t1n0e0, tile2d_launch_t2n0e0},
     {tile2d_launch_t0n1e0, tile2d_launch_t1n1e0, tile2d_launch_t2n1e0}},
    {{tile2d_launch_t0n0e1, tile2d_launch_t1n0e1, tile2d_launch_t2n0e1},
     {tile2d_launch_t0n1e1, tile2d_launch_t1n1e1, tile2d_launch_t2n1e1}}};

bool tier_ok(int tier) { return tier >= 0 && tier < kNumTiers; }

// Tile rows the producer of a plain 2-D launch walks together (measured on
// GB300, strided_bf16 A/B on one box: 1 -> 5982 GB/s, 8 -> 6076; 4 and 16
// less than 8, 32 below 1).
constexpr uint32_t kTileGroupRows = 8;

}  // namespace

cudaError_t upload_program(int tier, bool ext, int slot, const uint32_t* words, int n) {
  if (!tier_ok(tier)) return cudaErrorInvalidValue;
  cudaError_t e = kContigUpload[ext][tier](slot, words, n);
  if (e == cudaSuccess && ext && tier == kTier2) e = contig_upload_t0e1o4(slot, words, n);
  if (e == cudaSuccess && !ext && tier == kTier4) e = contig_upload_t1e0h16(slot, words, n);
  if (e == cudaSuccess) e = kGenericUpload[ext][tier](slot, words, n);
  for (int nd = 0; nd < 2 && e == cudaSuccess && !tier_wide(tier); ++nd) e = kTileUpload[ext][nd][tier](slot, words, n);
  return e;
}

cudaError_t contig_launch(int tier, bool ext, const ContigParams& p, cudaStream_t stream, bool bits_only,
                          bool half2) {
  if (!tier_ok(tier)) return cudaErrorInvalidValue;
  if (half16(tier, ext, half2)) return contig_launch_t1e0h16(p, stream);
  if (ext && tier == kTier2 && bits_only) return contig_launch_t0e1o4(p, stream);
  return kContigLaunch[ext][tier](p, stream);
}

cudaError_t generic_launch(int tier, bool ext, const GenericParams& p, cudaStream_t stream) {
  if (!tier_ok(tier)) return cudaErrorInvalidValue;
  return kGenericLaunch[ext][tier](p, stream);
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

cudaError_t tile2d_launch(int tier, bool ext, const Tile2dLaunch& L, cudaStream_t stream) {
  static_assert(sizeof(Tile2dParams) < 8192, "kernel parameters stay small");
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  Tile2dParams p;
  std::memset(&p, 0, sizeof p);
  uint32_t off = 0, tx = 0;
  // a batched launch: batch dims or broadcast loads (it runs the ND kernel)
  bool batched = L.nb[0] > 1 || L.nb[1] > 1;
  for (uint32_t j = 0; j < L.n_loads; ++j)
    batched = batched || L.in_ld[j] == 0 || L.in_bst[j][0] != 0 || L.in_bst[j][1] != 0;
  for (uint32_t j = 0; j < L.n_loads; ++j) {
    const bool half = L.in_dt[j] == 1 || L.in_dt[j] == 2;
    const uint32_t es = half ? 2 : 4;
    const bool trans = L.in_trans[j] != 0;
    // descriptor dims: 0 = the unit-stride tile dim; then the other tile dim
    // and the batch dims that have a nonzero stride, by increasing stride.
    // A transposed load whose column count is a multiple of 8 has its column
    // dim split in two, (column / 8, stride 8 ld) then (column % 8, stride
    // ld), each a box of 8: column 8 g + k then lands in box row g + 8 k,
    // which the consumers read without bank conflicts or register permutes.
    // Measured on GB300 it pays for 4-byte loads in batched launches of the
    // 2-slot tier (+5% against rotated reads, +1.2% against XOR-order ones);
    // a 2-byte load with 16 KB rows ran 15% slower split (the box then walks
    // rows eight apart), and the extra read path cost the plain 2-D kernel
    // 3%, so only that case splits.
    struct D { int64_t stride, size; int src; uint32_t box; };
    auto encode_load = [&](bool split) -> CUresult {
      D d[4];
      int nd = 0;
      if (split) {
        d[nd++] = {8 * L.in_ld[j], L.cols / 8, 3, 8};
        d[nd++] = {L.in_ld[j], 8, 4, 8};
      } else if (L.in_ld[j] != 0) {
        d[nd++] = {L.in_ld[j], trans ? L.cols : L.rows, 0, 64};
      }
      const int first_sorted = split ? nd : 0;  // the split pair keeps its order
      if (L.in_bst[j][0] != 0) d[nd++] = {L.in_bst[j][0], L.nb[0], 1, 1};
      if (L.in_bst[j][1] != 0) d[nd++] = {L.in_bst[j][1], L.nb[1], 2, 1};
      for (int a = first_sorted + 1; a < nd; ++a)
        for (int b = a; b > first_sorted && d[b].stride < d[b - 1].stride; --b) std::swap(d[b], d[b - 1]);
      cuuint64_t dims[5] = {(cuuint64_t)(trans ? L.rows : L.cols), 1, 1, 1, 1};
      cuuint64_t strides[4] = {0, 0, 0, 0};
      cuuint32_t box[5] = {half ? 64u : 32u, 1, 1, 1, 1};
      cuuint32_t estr[5] = {1, 1, 1, 1, 1};
      for (int k = 0; k < 4; ++k) p.in_src[j][k] = 0;
      for (int k = 0; k < nd; ++k) {
        dims[k + 1] = (cuuint64_t)d[k].size;
        strides[k] = (cuuint64_t)d[k].stride * es;
        box[k + 1] = d[k].box;
        p.in_src[j][k] = (uint8_t)d[k].src;
      }
      const int rank = 1 + nd;
      p.in_rank[j] = (uint8_t)rank;
      p.in_split[j] = split ? 1 : 0;
      return encode(&p.maps[j], half ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32,
                    (cuuint32_t)rank, const_cast<void*>(L.in[j]), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    const bool can_split = batched && !half && tier == kTier2 && trans && L.in_ld[j] != 0 && L.cols % 8 == 0;
    CUresult r = can_split ? encode_load(true) : CUDA_ERROR_INVALID_VALUE;
    if (r != CUDA_SUCCESS) r = encode_load(false);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    p.in_bcast[j] = L.in_ld[j] == 0;
    p.load_off[j] = off;
    off += (uint32_t)tile_stage_bytes((int)es);
    // bytes the load's boxes deliver per tile: one row when broadcast
    tx += (uint32_t)(p.in_bcast[j] ? 64 * es : 64 * 64 * es);
    p.in_dt[j] = L.in_dt[j];
    p.in_trans[j] = L.in_trans[j];
  }
  if (off == 0 || off > (uint32_t)kTileStageLimit) return cudaErrorInvalidValue;
  p.stage_bytes = off;
  p.tx_bytes = tx;
  // stages within 48 KB for the 2-slot tier (its kernel is built for four
  // CTAs per SM: 3 stages of two 2-byte loads; measured against 4 stages at
  // three CTAs, strided_bf16 +4%, and two 4-byte loads 2 stages at three
  // CTAs against 3 at two, batched_transpose +8%), 96 KB for the others
  const uint32_t stages_fit = (uint32_t)((tier == kTier2 ? 1 : 2) * kTileStageLimit / off);
  p.n_stages = stages_fit < 2 ? 2 : stages_fit > kMaxStages ? kMaxStages : stages_fit;
  for (int j = 0; j < kMaxStores; ++j) {
    p.out[j] = L.out[j];
    p.out_ld[j] = L.out_ld[j];
    p.out_bst[j][0] = L.out_bst[j][0];
    p.out_bst[j][1] = L.out_bst[j][1];
  }
  std::memcpy(p.scal, L.scal, sizeof p.scal);
  p.err = L.err;
  p.rows = L.rows;
  p.cols = L.cols;
  p.tiles_c = (uint32_t)((L.cols + kTileCols - 1) / kTileCols);
  p.tiles_r = (uint32_t)((L.rows + kTileRows - 1) / kTileRows);
  p.nb1 = (uint32_t)L.nb[1];
  p.n_tiles = (uint32_t)((int64_t)p.tiles_c * p.tiles_r * L.nb[0] * L.nb[1]);
  p.group_rows = kTileGroupRows < p.tiles_r ? kTileGroupRows : (p.tiles_r > 0 ? p.tiles_r : 1);
  p.timeout_ns = L.timeout_ns;
  p.prog = L.prog;
  p.n_loads = L.n_loads;
  p.debug = L.debug;
  bool nd = L.nb[0] > 1 || L.nb[1] > 1;
  for (uint32_t j = 0; j < L.n_loads; ++j) nd = nd || p.in_bcast[j] || p.in_rank[j] != 2;
  if (tier < kTier2 || tier > kTier8) return cudaErrorInvalidValue;  // no wide-tier tile kernel
  return kTileLaunch[ext][nd][tier](p, stream);
}

}  // namespace cmdx
