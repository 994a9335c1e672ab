// mxfp8.cu -- MXFP8 quantisers for the fp8_bwd backward (E4M3 values, one
// UE8M0 power-of-two scale per 32 consecutive elements along a GEMM's K).
//
// MXFP8 block scaling on Blackwell and group-aware quantisation are named in
// the NVIDIA MoE article ("Que optimizaciones especificas exige el MoE sin
// descartes": MXFP8 group quantisation, MXFP8 grouped GEMM); the fp8_bwd mode
// (BF16 forward, FP8 backward) in the Prime Mega MoE write-ups.
//
// The scale rule and the E4M3 conversion are in mxfp8.cuh (shared with the
// block-scaled dA GEMM, whose epilogue quantises dG and dU itself).
//
// Output layouts are what the block-scaled tensor-core GEMM loads:
//   codes  K-major: [rows][K] bytes;
//   scales in 512-byte atoms of 128 rows x 128 K: atom (rb, kg) at
//          ((rb * (K / 128)) + kg) * 512 holds the scale of its row 32 q + l
//          and K block kg*4 + j at byte l*16 + q*4 + j -- the layout
//          tcgen05.cp.32x128b.warpx4 copies into tensor memory for the MMA.
//          Rows map to row blocks rb by an SfLayout: rows are cut into segments
//          of `seg` rows (an expert's rows of a weight, or the whole operand),
//          each segment into groups of `group` rows (128, or 192 for the
//          GEMMs' 192-row B tiles), each group into ceil(group/128) atoms, so a
//          tile's scales always start on an atom boundary.
// Ragged operands are written in a per-expert padded row space: expert e's
// rows start at pad_off[e] = sum over e' < e of ceil(count/128)*128, the rows
// past its count are zero codes with zero scales, so every 128-row tile and
// every 32-element block along tokens starts inside one expert.
#include "mxfp8.cuh"

namespace moe {
namespace {

// Expert of padded row o (largest e with pad_off[e] <= o), from shared memory.
__device__ __forceinline__ int expert_of(int o, const int *s_pad, int E) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pad[mid] <= o)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// The transposing quantisers stage 128 x 64 bf16 tiles in shared memory by
// cp.async (16-byte chunks XOR-swizzled by row, so that both a column walk and
// a row walk are free of bank conflicts), several tiles in flight per block.
// Along the tiles' columns one thread per (column, 32-row block) quantises
// down the column into a shared output tile (64 rows of 128 codes, rows padded
// to 144 bytes against bank conflicts), which leaves as full 128-byte rows:
// the codes of an operand whose reduction axis is the tiles' row axis, written
// transposed.  Along the rows one thread per (row, 32-column block) quantises
// straight from the staged tile.  Every address a thread uses is fixed up to
// the tile's column offset, so it is computed once per block: a thread stages
// 16-byte piece (tid mod 8) of rows tid/8 + 32 j of each tile (absent rows
// zero-filled by the copy itself), reads row tid/2 in the row pass and column
// tid mod 64 in the column pass, and stores 16-byte piece (tid mod 8) of output
// rows tid/8 + 32 j.
constexpr int kQcRows = 128, kQcCols = 64, kQcThreads = 256;
constexpr int kQcRing = 4;                                  // staged tiles in flight per block
constexpr int kQcTileElems = kQcRows * kQcCols;             // bf16 per staged tile
constexpr int kQcTileBytes = kQcTileElems * 2;              // 16 KB
constexpr int kQcOutStride = kQcRows + 16;                  // bytes per output row in shared memory
constexpr int kQcSmem = kQcRing * kQcTileBytes + kQcCols * kQcOutStride;  // dynamic shared memory
constexpr int kQcLoads = (kQcRows * kQcCols / 8) / kQcThreads;   // 16-byte pieces staged per thread per tile
constexpr int kQcStores = (kQcCols * kQcRows / 16) / kQcThreads;  // 16-byte code pieces stored per thread per tile
static_assert(kQcLoads == 4 && kQcStores == 2, "thread shares assume 256 threads and 128 x 64 tiles");

// 16-byte cp.async; with src_bytes 0 nothing is read and the 16 bytes are zeroed.
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most n of this thread's cp.async groups are still pending (n < 4).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  if (n <= 0)
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  else if (n == 1)
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  else if (n == 2)
    asm volatile("cp.async.wait_group 2;" ::: "memory");
  else
    asm volatile("cp.async.wait_group 3;" ::: "memory");
}

// A thread's share of staging a tile: row tid/8 + 32 j (j < 4) of the source
// starts at src[j] (its piece's column offset included), or is absent
// (bytes[j] = 0: zero-filled, src[j] any readable address).
struct QcStage {
  const uint16_t *src[kQcLoads];
  uint32_t bytes[kQcLoads];
  uint32_t soff;  // byte offset of the thread's piece of row tid/8 in a tile
};
template <class RowPtr>
__device__ __forceinline__ QcStage qc_stage_plan(const RowPtr &row_ptr, const uint16_t *readable) {
  QcStage p;
  const int lr = threadIdx.x >> 3, part = threadIdx.x & 7;
  p.soff = static_cast<uint32_t>(lr * kQcCols + ((part ^ (lr & 7)) << 3)) * 2;
#pragma unroll
  for (int j = 0; j < kQcLoads; ++j) {
    const uint16_t *s = row_ptr(lr + 32 * j);  // nullptr: absent row
    p.src[j] = (s ? s : readable) + part * 8;
    p.bytes[j] = s ? 16u : 0u;
  }
  return p;
}
// Issue the thread's copies of columns c0 .. c0 + 63 into the tile at shared address tile.
__device__ __forceinline__ void qc_stage(const QcStage &p, uint32_t tile, int c0) {
#pragma unroll
  for (int j = 0; j < kQcLoads; ++j) cp_async16(tile + p.soff + j * (32 * kQcCols * 2), p.src[j] + c0, p.bytes[j]);
}

// Element (r, c) of a staged tile.
__device__ __forceinline__ int qc_idx(int r, int c) { return r * kQcCols + (((c >> 3) ^ (r & 7)) << 3) + (c & 7); }

// 32 bf16 values of a staged tile: row r, columns 32 bb .. 32 bb + 31.
__device__ __forceinline__ void qc_row32(const uint16_t *tile, int r, int bb, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = *reinterpret_cast<const uint4 *>(tile + r * kQcCols + (((4 * bb + q) ^ (r & 7)) << 3));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * q + 2 * h] = bf16_lo(ww[h]);
      v[8 * q + 2 * h + 1] = bf16_hi(ww[h]);
    }
  }
}

// 32 bf16 values of a staged tile down column c: rows 32 b .. 32 b + 31.
__device__ __forceinline__ void qc_col32(const uint16_t *tile, int c, int b, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(static_cast<uint32_t>(tile[qc_idx(32 * b + i, c)]) << 16);
}

// The column-tile walk shared by the transposing quantisers: tiles c0 = first,
// first + step, ... < C through a ring of kRing slots of slot_bytes, kRing - 1
// issued ahead; stage(slot address, c0) issues one tile's copies (one group);
// work(slot, c0) runs once the tile has landed, after a block barrier.  A slot
// is staged again at the top of the iteration after the one that read it, so
// work must finish its reads of the slot before a block barrier of its own,
// or ask for a trailing barrier (trail).
template <int kRing, class Stage, class Work>
__device__ __forceinline__ void qc_walk(uint8_t *ring, int slot_bytes, int first, int step, int C, bool trail,
                                        const Stage &stage, const Work &work) {
  const int nt = first < C ? (C - first + step - 1) / step : 0;
  const uint32_t ring_s = smem_addr(ring);
  for (int i = 0; i < kRing - 1 && i < nt; ++i) {
    stage(ring_s + i * slot_bytes, first + i * step);
    cp_async_commit();
  }
  int slot = 0;
  for (int it = 0; it < nt; ++it) {
    const int ahead = it + kRing - 1;
    if (ahead < nt) {  // into the slot read in the previous iteration
      stage(ring_s + (slot == 0 ? kRing - 1 : slot - 1) * slot_bytes, first + ahead * step);
      cp_async_commit();
    }
    cp_async_wait_pending(min(nt - 1, ahead) - it);  // this tile's group has landed
    __syncthreads();
    work(ring + slot * slot_bytes, first + it * step);
    if (trail) __syncthreads();
    slot = slot + 1 == kRing ? 0 : slot + 1;
  }
}

// Token-axis quantisation, output transposed: codes [C][Mpad] (tokens
// contiguous), scales grouped by 128 (one segment: L.seg >= C).  A block takes
// 128 padded rows (one expert's, as segments are 128-aligned) and walks their
// columns; the rows may be gathered from a token-major source (permuted row r
// reads token slot_of_row[r] / k) instead of read from a permuted copy, and
// the gathered rows may be written out in bf16 as well (the permuted copy
// itself, xp); codes may be null (xp only).  Tiles past the padded total are
// skipped.
__global__ void __launch_bounds__(kQcThreads, 3) quant_cols_kernel(const uint16_t *__restrict__ src, int C,
                                                                int Mpad,
                                                                const int32_t *__restrict__ offsets,
                                                                const int32_t *__restrict__ pad_off, int E,
                                                                uint8_t *__restrict__ codes,
                                                                uint8_t *__restrict__ sf,
                                                                const int32_t *__restrict__ slot_of_row, int k,
                                                                uint16_t *__restrict__ xp) {
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) uint8_t qc_smem[];
  uint8_t *otile = qc_smem + kQcRing * kQcTileBytes;
  __shared__ int s_pad[kMaxExperts + 1];
  __shared__ int s_seg[3];  // first source row, valid rows of this tile, skip flag
  const int prow0 = blockIdx.x * kQcRows;
  for (int e = threadIdx.x; e <= E; e += kQcThreads) s_pad[e] = __ldg(pad_off + e);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (prow0 >= s_pad[E]) {
      s_seg[2] = 1;
    } else {
      const int e = expert_of(prow0, s_pad, E);
      const int o = __ldg(offsets + e), count = __ldg(offsets + e + 1) - o;
      const int local0 = prow0 - s_pad[e];
      s_seg[0] = o + local0;
      s_seg[1] = min(kQcRows, count - local0);
      s_seg[2] = 0;
    }
  }
  __syncthreads();
  if (s_seg[2]) return;
  const int row0 = s_seg[0], nvalid = s_seg[1];
  __shared__ int s_src[kQcRows];  // source row of each permuted row (its token's, when gathering)
  for (int r = threadIdx.x; r < nvalid; r += kQcThreads)
    s_src[r] = slot_of_row ? __ldg(slot_of_row + row0 + r) / k : row0 + r;
  __syncthreads();
  const QcStage ld = qc_stage_plan(
      [&](int r) -> const uint16_t * { return r < nvalid ? src + static_cast<size_t>(s_src[r]) * C : nullptr; }, src);
  const int lr = threadIdx.x >> 3, part = threadIdx.x & 7;  // staged pieces (and xp's)
  uint16_t *xrow = xp ? xp + static_cast<size_t>(row0 + lr) * C + part * 8 : nullptr;
  const int cc = threadIdx.x % kQcCols, b = threadIdx.x / kQcCols;  // column pass: column, 32-token block
  uint8_t *csf = sf + atom_kblock((prow0 >> 5) + b);
  uint8_t *obase = codes ? codes + static_cast<size_t>(lr) * Mpad + prow0 + part * 16 : nullptr;
  const uint8_t *osrc = otile + lr * kQcOutStride + part * 16;
  qc_walk<kQcRing>(
      qc_smem, kQcTileBytes, blockIdx.y * kQcCols, gridDim.y * kQcCols, C, codes == nullptr,
      [&](uint32_t tile, int c0) { qc_stage(ld, tile, c0); },
      [&](const uint8_t *slot, int c0) {
        const uint16_t *tile = reinterpret_cast<const uint16_t *>(slot);
        if (xp) {  // the staged rows in bf16: 16-byte pieces, 128 bytes per row
#pragma unroll
          for (int j = 0; j < kQcLoads; ++j)
            if (lr + 32 * j < nvalid)
              *reinterpret_cast<uint4 *>(xrow + static_cast<size_t>(32 * j) * C + c0) =
                  *reinterpret_cast<const uint4 *>(slot + ld.soff + j * (32 * kQcCols * 2));
        }
        if (codes) {  // along the tokens, transposed
          float v[32];
          qc_col32(tile, cc, b, v);
          csf[atom_row_sg<128>(0, c0 + cc, Mpad, C)] =
              quant32(v, reinterpret_cast<uint4 *>(otile + cc * kQcOutStride + 32 * b));
          __syncthreads();  // the output tile is complete; the staged tile is no longer read
          uint8_t *o = obase + static_cast<size_t>(c0) * Mpad;
#pragma unroll
          for (int j = 0; j < kQcStores; ++j)
            *reinterpret_cast<uint4 *>(o + static_cast<size_t>(32 * j) * Mpad) =
                *reinterpret_cast<const uint4 *>(osrc + 32 * j * kQcOutStride);
        }
      });
}

// The MXFP8 backward's pass over dy (one read, no bf16 copy): for 128 padded
// rows of one expert (a block) and 64-column tiles of H, the rows of dy the
// permuted rows come from (gathered by token: slot_of_row / k) and the same
// rows of Y are staged by cp.async, kDyRing tiles of each in flight.  Each
// tile is quantised along H (thread = row, 32-column block; into the padded
// row space, scales grouped by 128 in one segment: dA's A operand) and along
// tokens (thread = column, 32-token block; transposed, scales grouped by kMxBN
// in one segment: dW_down's B operand), and every row accumulates its part of
// g = <dy_t, Y_r> over the block's columns; the part of block column y of row
// r goes to g_part[r * gridDim.y + y], added in order by the router gradient
// kernel.  Two tile pairs in a ring (one in flight while the other is
// quantised) keep the block at 73 KB and 80 registers, three blocks per SM:
// measured faster than three pairs at two blocks per SM.
constexpr int kDyRing = 2;
constexpr int kDySmem = kDyRing * 2 * kQcTileBytes + kQcCols * kQcOutStride;

__global__ void __launch_bounds__(kQcThreads, 3) dy_quant_kernel(const uint16_t *__restrict__ dy,
                                                                 const uint16_t *__restrict__ Y,
                                                                 const int32_t *__restrict__ slot_of_row, int k,
                                                                 int H, int Mpad, const int32_t *__restrict__ offsets,
                                                                 const int32_t *__restrict__ pad_off, int E,
                                                                 uint8_t *__restrict__ codes_t, uint8_t *__restrict__ sf_t,
                                                                 uint8_t *__restrict__ codes, uint8_t *__restrict__ sf,
                                                                 float *__restrict__ g_part) {
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) uint8_t qc_smem[];
  uint8_t *otile = qc_smem + kDyRing * 2 * kQcTileBytes;
  __shared__ int s_pad[kMaxExperts + 1];
  __shared__ int s_seg[3];  // first source row, valid rows of this tile, skip flag
  __shared__ int s_tok[kQcRows];
  const int prow0 = blockIdx.x * kQcRows;
  for (int e = threadIdx.x; e <= E; e += kQcThreads) s_pad[e] = __ldg(pad_off + e);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (prow0 >= s_pad[E]) {
      s_seg[2] = 1;
    } else {
      const int e = expert_of(prow0, s_pad, E);
      const int o = __ldg(offsets + e), count = __ldg(offsets + e + 1) - o;
      const int local0 = prow0 - s_pad[e];
      s_seg[0] = o + local0;
      s_seg[1] = min(kQcRows, count - local0);
      s_seg[2] = 0;
    }
  }
  __syncthreads();
  if (s_seg[2]) return;
  const int row0 = s_seg[0], nvalid = s_seg[1];
  for (int r = threadIdx.x; r < nvalid; r += kQcThreads) s_tok[r] = __ldg(slot_of_row + row0 + r) / k;
  __syncthreads();
  const QcStage ldy = qc_stage_plan(
      [&](int r) -> const uint16_t * { return r < nvalid ? dy + static_cast<size_t>(s_tok[r]) * H : nullptr; }, dy);
  const QcStage ly = qc_stage_plan(
      [&](int r) -> const uint16_t * { return r < nvalid ? Y + static_cast<size_t>(row0 + r) * H : nullptr; }, Y);
  const int r = threadIdx.x >> 1, bb = threadIdx.x & 1;  // row pass: row, 32-column block
  uint8_t *rcodes = codes + static_cast<size_t>(prow0 + r) * H + 32 * bb;
  uint8_t *rsf = sf + atom_row_sg<128>(0, prow0 + r, H, Mpad);
  const int cc = threadIdx.x % kQcCols, b = threadIdx.x / kQcCols;  // column pass: column, 32-token block
  uint8_t *csf = sf_t + atom_kblock((prow0 >> 5) + b);
  const int orow = threadIdx.x >> 3, opart = threadIdx.x & 7;  // output pieces
  uint8_t *obase = codes_t + static_cast<size_t>(orow) * Mpad + prow0 + opart * 16;
  const uint8_t *osrc = otile + orow * kQcOutStride + opart * 16;
  float gpart = 0.f;
  qc_walk<kDyRing>(
      qc_smem, 2 * kQcTileBytes, blockIdx.y * kQcCols, gridDim.y * kQcCols, H, false,
      [&](uint32_t tile, int c0) {  // one group per tile: both sources
        qc_stage(ldy, tile, c0);
        qc_stage(ly, tile + kQcTileBytes, c0);
      },
      [&](const uint8_t *slot, int c0) {
        const uint16_t *tile = reinterpret_cast<const uint16_t *>(slot), *ytile = tile + kQcTileElems;
        {
          float v[32], yv[32];
          qc_row32(tile, r, bb, v);
          qc_row32(ytile, r, bb, yv);
#pragma unroll
          for (int i = 0; i < 32; ++i) gpart = fmaf(v[i], yv[i], gpart);
          rsf[atom_kblock((c0 >> 5) + bb)] = quant32(v, reinterpret_cast<uint4 *>(rcodes + c0));
        }
        float v[32];
        qc_col32(tile, cc, b, v);
        csf[atom_row_sg<kMxBN>(0, c0 + cc, Mpad, H)] =
            quant32(v, reinterpret_cast<uint4 *>(otile + cc * kQcOutStride + 32 * b));
        __syncthreads();  // the output tile is complete; the staged tiles are no longer read
        uint8_t *o = obase + static_cast<size_t>(c0) * Mpad;
#pragma unroll
        for (int j = 0; j < kQcStores; ++j)
          *reinterpret_cast<uint4 *>(o + static_cast<size_t>(32 * j) * Mpad) =
              *reinterpret_cast<const uint4 *>(osrc + 32 * j * kQcOutStride);
      });
  gpart += __shfl_xor_sync(0xffffffffu, gpart, 1);  // the row's two 32-column halves
  if (bb == 0 && r < nvalid) g_part[static_cast<size_t>(row0 + r) * gridDim.y + blockIdx.y] = gpart;
}

// Weights quantised along their middle axis (the mxfp8 forward GEMMs' K),
// written transposed: W [E, R, C] bf16 (R the reduction axis, R % 128 == 0)
// -> codes [rows, R] with output row (e, c) = e * C + c (W_down: the down
// GEMM's B rows), or, interleaved for gate|up tiles, e * 2C + (c / 32) * 64 +
// half * 32 + c % 32 (W_gate half 0, W_up half 1: every 64 B rows hold 32
// gate columns then the same 32 up columns); scales grouped by kMxBN in
// segments of one expert's output rows.  Optionally the same staged tile is
// also quantised along C, row by row (the backward GEMMs' weight operand,
// codes [E * R, C], scales grouped by kMxBN in segments of R rows), so each
// weight is read once for both.  A block takes 128 rows of one expert.
__global__ void __launch_bounds__(kQcThreads, 3) quant_wT_kernel(const uint16_t *__restrict__ src, int R,
                                                                 int C, int interleave, int half,
                                                                 uint8_t *__restrict__ codes,
                                                                 uint8_t *__restrict__ sf, int seg,
                                                                 uint8_t *__restrict__ rcodes_all,
                                                                 uint8_t *__restrict__ rsf_all) {
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) uint8_t qc_smem[];
  uint8_t *otile = qc_smem + kQcRing * kQcTileBytes;
  const int grow0 = blockIdx.x * kQcRows;  // first source row (of E * R)
  const int e = grow0 / R, r0 = grow0 - e * R;
  const QcStage ld = qc_stage_plan(
      [&](int r) -> const uint16_t * { return src + static_cast<size_t>(grow0 + r) * C; }, src);
  const int r = threadIdx.x >> 1, bb = threadIdx.x & 1;  // row pass: row, 32-column block
  uint8_t *rcodes = rcodes_all ? rcodes_all + static_cast<size_t>(grow0 + r) * C + 32 * bb : nullptr;
  uint8_t *rsf = rsf_all ? rsf_all + atom_row_sg<kMxBN>(e, r0 + r, C, R) : nullptr;
  const int cc = threadIdx.x % kQcCols, b = threadIdx.x / kQcCols;  // column pass: column, 32-row block
  uint8_t *csf = sf + atom_kblock((r0 >> 5) + b);
  const int orow = threadIdx.x >> 3, opart = threadIdx.x & 7;  // output pieces
  const uint8_t *osrc = otile + orow * kQcOutStride + opart * 16;
  // output row of column c within the expert's segment
  auto seg_row = [&](int c) { return interleave ? (c >> 5) * 64 + half * 32 + (c & 31) : c; };
  qc_walk<kQcRing>(
      qc_smem, kQcTileBytes, blockIdx.y * kQcCols, gridDim.y * kQcCols, C, false,
      [&](uint32_t tile, int c0) { qc_stage(ld, tile, c0); },
      [&](const uint8_t *slot, int c0) {
        const uint16_t *tile = reinterpret_cast<const uint16_t *>(slot);
        if (rcodes) {  // along C: thread = (row, 32-column block)
          float v[32];
          qc_row32(tile, r, bb, v);
          rsf[atom_kblock((c0 >> 5) + bb)] = quant32(v, reinterpret_cast<uint4 *>(rcodes + c0));
        }
        float v[32];
        qc_col32(tile, cc, b, v);
        csf[atom_row_sg<kMxBN>(e, seg_row(c0 + cc), R, seg)] =
            quant32(v, reinterpret_cast<uint4 *>(otile + cc * kQcOutStride + 32 * b));
        __syncthreads();  // the output tile is complete; the staged tile is no longer read
        // output rows c0 + orow + 32 j: (c >> 5) = (c0 >> 5) + j and c % 32 = orow, c0 being a multiple of 64
        const size_t orow0 = static_cast<size_t>(e) * seg + seg_row(c0 + orow);
        uint8_t *o = codes + orow0 * R + r0 + opart * 16;
        const size_t jstride = static_cast<size_t>(interleave ? 64 : 32) * R;
#pragma unroll
        for (int j = 0; j < kQcStores; ++j)
          *reinterpret_cast<uint4 *>(o + j * jstride) = *reinterpret_cast<const uint4 *>(osrc + 32 * j * kQcOutStride);
      });
}

// pad_off[e] = sum over e' < e of ceil(count/128)*128; pad_off[E] = padded total.
__global__ void __launch_bounds__(32) pad_offsets_kernel(const int32_t *__restrict__ offsets, int E,
                                                         int32_t *__restrict__ pad_off) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int lane = threadIdx.x;
  int carry = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const int c = e < E ? ((offsets[e + 1] - offsets[e] + 127) / 128) * 128 : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (e < E) pad_off[e] = carry + incl - c;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) pad_off[E] = carry;
}

}  // namespace

cudaError_t launch_pad_offsets(const int32_t *offsets, int E, int32_t *pad_off, cudaStream_t s) {
  return launch_pdl(pad_offsets_kernel, dim3(1), dim3(32), 0, s, 1, offsets, E, pad_off);
}

cudaError_t launch_quant_cols(const uint16_t *src, int C, int Mpad, const int32_t *offsets,
                              const int32_t *pad_off, int E, uint8_t *codes, uint8_t *sf, SfLayout L,
                              cudaStream_t s, const int32_t *slot_of_row, int k, uint16_t *xp) {
  if (codes && (L.group != 128 || L.seg < C)) return cudaErrorInvalidValue;  // one segment, groups of 128
  const int col_blocks = C / kQcCols < 4 ? C / kQcCols : 4;  // each loops over C / (64 * 4) column tiles
  const dim3 grid(static_cast<unsigned>(Mpad / kQcRows), static_cast<unsigned>(col_blocks));
  static DeviceOnce once;  // dynamic shared memory above 48 KB, opted in once per device
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(quant_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQcSmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(quant_cols_kernel, grid, dim3(kQcThreads), kQcSmem, s, 1, src, C, Mpad, offsets, pad_off, E,
                    codes, sf, slot_of_row, k, xp);
}

cudaError_t launch_dy_quant(const uint16_t *dy, const uint16_t *Y, const int32_t *slot_of_row, int k, int H,
                            int Mpad, const int32_t *offsets, const int32_t *pad_off, int E, uint8_t *codes_t,
                            uint8_t *sf_t, SfLayout Lt, RowCodes rows, float *g_part, int col_blocks,
                            cudaStream_t s) {
  // both scale buffers in one segment: transposed grouped by kMxBN, rows by 128
  if (Lt.group != kMxBN || Lt.seg < H || rows.L.group != 128 || rows.L.seg < Mpad || !rows.codes)
    return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(Mpad / kQcRows), static_cast<unsigned>(col_blocks));
  static DeviceOnce once;  // dynamic shared memory above 48 KB, opted in once per device
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(dy_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDySmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(dy_quant_kernel, grid, dim3(kQcThreads), kDySmem, s, 1, dy, Y, slot_of_row, k, H, Mpad, offsets,
                    pad_off, E, codes_t, sf_t, rows.codes, rows.sf, g_part);
}

int dy_quant_col_blocks(int H) { return H / kQcCols < 4 ? H / kQcCols : 4; }

cudaError_t launch_quant_wT(const uint16_t *W, int E, int R, int C, int interleave, int half,
                            uint8_t *codes, uint8_t *sf, SfLayout L, RowCodes rows, cudaStream_t s) {
  // scales grouped by kMxBN in per-expert segments: the transposed codes' of the
  // expert's output rows, the row codes' of its R rows
  if (L.group != kMxBN || L.seg != (interleave ? 2 * C : C) ||
      (rows.codes && (rows.L.group != kMxBN || rows.L.seg != R)))
    return cudaErrorInvalidValue;
  // one block walks all of its 128 rows' column tiles (measured faster than
  // splitting them over 2 or 4 blocks: 12-tile walks instead of 3- or 6-tile ones
  // at the 30B shape's I = 768)
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(E) * R / kQcRows), 1);
  static DeviceOnce once;
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(quant_wT_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQcSmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(quant_wT_kernel, grid, dim3(kQcThreads), kQcSmem, s, 1, W, R, C, interleave, half, codes, sf,
                    L.seg, rows.codes, rows.sf);
}

}  // namespace moe
