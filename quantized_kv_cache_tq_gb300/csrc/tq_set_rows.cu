// SET_ROWS: quantise-on-write of K/V rows into the packed TurboQuant cache
// ([TQ#36] "shuffle WHT"; the per-block arithmetic is in tq_quant.cuh).
// The page's kernel holds one element per thread, so it needs shuffles for
// h = 1..16 and barriers for h = 32, 64; here four lanes own a block and only
// h = 4, 8 cross lanes (~11 warp shuffles per block, one warp per 8 blocks).
#include "tq_quant.cuh"

namespace tq {
namespace {

template <int TYPE, int SRC>
__global__ void __launch_bounds__(256) set_rows_kernel(const SetRowsArgs a) {
  constexpr int QSB = TypeTraits<TYPE>::QSB;
  const int lane = threadIdx.x & 31;
  const int l4 = lane & 3;                     // position inside the block's 4 lanes
  const int64_t total = a.n_rows * a.n_kv_heads * a.n_blocks;
  const int64_t blk_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
  const bool active = blk_id < total;          // whole 4-lane groups are active or not

  int b = 0, h = 0;
  int64_t row = 0, cell = 0;
  bool ok = false;
  float v[8][4];
  if (active) {
    if (total <= 0x7fffffff) {                 // 32-bit division when the ids fit
      const uint32_t id = static_cast<uint32_t>(blk_id), nb = a.n_blocks, nh = a.n_kv_heads;
      const uint32_t rh = id / nb;
      b = static_cast<int>(id - rh * nb);
      row = rh / nh;
      h = static_cast<int>(rh - static_cast<uint32_t>(row) * nh);
    } else {
      b = static_cast<int>(blk_id % a.n_blocks);
      const int64_t rh = blk_id / a.n_blocks;
      h = static_cast<int>(rh % a.n_kv_heads);
      row = rh / a.n_kv_heads;
    }
    cell = a.cell_ids[row];
    ok = cell >= 0 && cell < a.n_cells;
    if (!ok && l4 == 0) set_status(a.dev_status, TQ_ERR_DEVICE_CHECK);
  }
  const int64_t base = (row * a.n_kv_heads + h) * a.head_dim + b * QK;
  const int valid = a.head_dim - b * QK;       // elements of the row from this block on
  if (ok && valid >= QK) {                     // a whole block: eight unconditional loads
#pragma unroll
    for (int i = 0; i < 8; ++i) quant_load4<SRC>(a.src, base + 4 * l4 + 16 * i, 4, v[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e0 = 4 * l4 + 16 * i;
      if (ok) quant_load4<SRC>(a.src, base + e0, valid - e0, v[i]);
      else v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
    }
  }

  // every lane takes part in the packing shuffles; only valid blocks store
  PackedShare<TYPE> pb;
  quantise_block4<TYPE>(a.cb, l4, v, pb);
  const int64_t blk = (static_cast<int64_t>(h) * a.n_cells + cell) * a.n_blocks + b;
  if (ok) store_block4<TYPE>(pb, l4, a.norms + blk, a.qs + blk * QSB, TYPE == 3 ? a.signs + blk * 16 : nullptr);
}

template <int TYPE>
cudaError_t launch_type(int src_type, const SetRowsArgs &a, cudaStream_t s) {
  const int64_t blocks = a.n_rows * a.n_kv_heads * a.n_blocks;
  const int64_t grid = (blocks * 4 + 255) / 256;
  switch (src_type) {
    case TQ_F32: set_rows_kernel<TYPE, TQ_F32><<<(unsigned)grid, 256, 0, s>>>(a); break;
    case TQ_F16: set_rows_kernel<TYPE, TQ_F16><<<(unsigned)grid, 256, 0, s>>>(a); break;
    default: set_rows_kernel<TYPE, TQ_BF16><<<(unsigned)grid, 256, 0, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_set_rows(int type, int src_type, const SetRowsArgs &a, cudaStream_t s) {
  switch (type) {
    case TQ_TURBO2: return launch_type<2>(src_type, a, s);
    case TQ_TURBO3: return launch_type<3>(src_type, a, s);
    default: return launch_type<4>(src_type, a, s);
  }
}

}  // namespace tq
