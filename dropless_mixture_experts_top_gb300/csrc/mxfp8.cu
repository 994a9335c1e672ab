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

// Token-axis quantisation, output transposed: codes [C][Mpad] (tokens
// contiguous).  A block takes 128 padded rows (one expert's, as segments are
// 128-aligned) and walks their columns in 64-wide tiles.  The tiles are staged
// in shared memory by cp.async, kQcRing of them in flight (16-byte chunks
// XOR-swizzled by row, so that both a column walk and a row walk are free of
// bank conflicts); one thread per (column, 32-token block) quantises down the
// column into a shared output tile (64 rows of 128 codes, rows padded to 144
// bytes against bank conflicts), which leaves as full 128-byte rows.
// Optionally the same tile is also quantised along its rows (one thread per
// (row, 32-column block)) into the padded row space, so an operand needed on
// both axes is read once; the rows may be gathered from a token-major source
// (permuted row r reads token slot_of_row[r] / k) instead of read from a
// permuted copy, and the gathered rows may be written out in bf16 as well (the
// permuted copy itself, xp).  Tiles past the padded total are skipped.
constexpr int kQcRows = 128, kQcCols = 64, kQcThreads = 256;
constexpr int kQcRing = 4;                         // staged tiles in flight per block
constexpr int kQcTileElems = kQcRows * kQcCols;   // bf16 per staged tile (16 KB)
constexpr int kQcOutStride = kQcRows + 16;         // bytes per output row in shared memory
constexpr int kQcSmem = kQcRing * kQcTileElems * 2 + kQcCols * kQcOutStride;  // dynamic shared memory
constexpr int kQcLoads = (kQcRows * kQcCols / 8) / kQcThreads;  // 16-byte pieces per thread per tile

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most n of this thread's cp.async groups are still pending (n < kQcRing).
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

// Element (r, c) of a staged tile.
__device__ __forceinline__ int qc_idx(int r, int c) { return r * kQcCols + (((c >> 3) ^ (r & 7)) << 3) + (c & 7); }

// Issue one 128 x 64 tile: source row r at row_ptr(r) (nullptr: a zero row),
// columns c0 .. c0 + 63; one cp.async group per call.
template <class RowPtr>
__device__ __forceinline__ void qc_issue(uint16_t *dst, int c0, const RowPtr &row_ptr, bool commit = true) {
#pragma unroll
  for (int j = 0; j < kQcLoads; ++j) {
    const int i = threadIdx.x + j * kQcThreads;
    const int r = i >> 3, part = i & 7;
    uint16_t *d = dst + r * kQcCols + ((part ^ (r & 7)) << 3);
    const uint16_t *sp = row_ptr(r);
    if (sp)
      cp_async16(d, sp + c0 + part * 8);
    else
      *reinterpret_cast<uint4 *>(d) = make_uint4(0, 0, 0, 0);
  }
  if (commit) cp_async_commit();
}

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

// The column-tile walk shared by both transposing quantisers: tiles c0 =
// first, first + step, ... < C, kQcRing - 1 of them issued ahead; work(tile,
// c0) runs on each once it has landed, between two block barriers.
template <class RowPtr, class Work>
__device__ __forceinline__ void qc_walk(uint16_t *ring, int first, int step, int C, const RowPtr &row_ptr,
                                        const Work &work) {
  const int nt = first < C ? (C - first + step - 1) / step : 0;
  for (int i = 0; i < kQcRing - 1 && i < nt; ++i) qc_issue(ring + i * kQcTileElems, first + i * step, row_ptr);
  for (int it = 0; it < nt; ++it) {
    const int ahead = it + kQcRing - 1;
    if (ahead < nt) qc_issue(ring + (ahead % kQcRing) * kQcTileElems, first + ahead * step, row_ptr);
    cp_async_wait_pending(min(nt - 1, ahead) - it);  // this tile's group has landed
    __syncthreads();
    work(ring + (it % kQcRing) * kQcTileElems, first + it * step);
    __syncthreads();  // the tile's slot and the output tile are reused
  }
}

__global__ void __launch_bounds__(kQcThreads, 3) quant_cols_kernel(const uint16_t *__restrict__ src, int C,
                                                                int Mpad,
                                                                const int32_t *__restrict__ offsets,
                                                                const int32_t *__restrict__ pad_off, int E,
                                                                uint8_t *__restrict__ codes,
                                                                uint8_t *__restrict__ sf, SfLayout L,
                                                                RowCodes rows,
                                                                const int32_t *__restrict__ slot_of_row, int k,
                                                                uint16_t *__restrict__ xp) {
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) uint8_t qc_smem[];
  uint16_t *ring = reinterpret_cast<uint16_t *>(qc_smem);
  uint8_t *otile = qc_smem + kQcRing * kQcTileElems * 2;
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
  auto row_ptr = [&](int r) -> const uint16_t * {
    return r < nvalid ? src + static_cast<size_t>(s_src[r]) * C : nullptr;
  };
  qc_walk(ring, blockIdx.y * kQcCols, gridDim.y * kQcCols, C, row_ptr, [&](const uint16_t *tile, int c0) {
    if (xp) {  // the staged rows in bf16: 16-byte pieces, 128 bytes per row
#pragma unroll
      for (int j = 0; j < kQcLoads; ++j) {
        const int i = threadIdx.x + j * kQcThreads;
        const int r = i >> 3, part = i & 7;
        if (r < nvalid)
          *reinterpret_cast<uint4 *>(xp + static_cast<size_t>(row0 + r) * C + c0 + part * 8) =
              *reinterpret_cast<const uint4 *>(tile + r * kQcCols + ((part ^ (r & 7)) << 3));
      }
    }
    if (rows.codes) {  // along the rows: thread = (row, 32-column block); zero rows past the count
      const int r = threadIdx.x >> 1, bb = threadIdx.x & 1;
      float v[32];
      qc_row32(tile, r, bb, v);
      const int prow = prow0 + r, kb = (c0 >> 5) + bb;
      rows.sf[atom_byte(prow, kb, C, rows.L)] =
          quant32(v, reinterpret_cast<uint4 *>(rows.codes + static_cast<size_t>(prow) * C + c0 + 32 * bb));
    }
    if (codes) {  // along the tokens, transposed
      const int cc = threadIdx.x % kQcCols, b = threadIdx.x / kQcCols;  // 4 blocks of 32 tokens
      float v[32];
      qc_col32(tile, cc, b, v);
      const size_t srow = L.group == 128 ? atom_row<128>(c0 + cc, Mpad, L) : atom_row(c0 + cc, Mpad, L);
      sf[srow + atom_kblock((prow0 >> 5) + b)] =
          quant32(v, reinterpret_cast<uint4 *>(otile + cc * kQcOutStride + 32 * b));
      __syncthreads();
#pragma unroll
      for (int j = 0; j < (kQcCols * kQcRows / 16) / kQcThreads; ++j) {
        const int i = threadIdx.x + j * kQcThreads;
        const int r = i >> 3, part = i & 7;  // output row (column c0 + r), 16-byte piece
        *reinterpret_cast<uint4 *>(codes + static_cast<size_t>(c0 + r) * Mpad + prow0 + part * 16) =
            *reinterpret_cast<const uint4 *>(otile + r * kQcOutStride + part * 16);
      }
    }
  });
}

// The MXFP8 backward's pass over dy (one read, no bf16 copy): for 128 padded
// rows of one expert (a block) and 64-column tiles of H, the rows of dy the
// permuted rows come from (gathered by token: slot_of_row / k) and the same
// rows of Y are staged by cp.async, kDyRing tiles of each in flight.  Each
// tile is quantised along H (thread = row, 32-column block; into the padded
// row space: dA's A operand) and along tokens (thread = column, 32-token
// block; transposed: dW_down's B operand), and every row accumulates its part
// of g = <dy_t, Y_r> over the block's columns; the part of block column
// y of row r goes to g_part[r * gridDim.y + y], added in order by the router
// gradient kernel.  The transposed codes' scale rows are grouped by kMxBN.
constexpr int kDyRing = 3;
constexpr int kDySmem = kDyRing * 2 * kQcTileElems * 2 + kQcCols * kQcOutStride;

__global__ void __launch_bounds__(kQcThreads, 2) dy_quant_kernel(const uint16_t *__restrict__ dy,
                                                                 const uint16_t *__restrict__ Y,
                                                                 const int32_t *__restrict__ slot_of_row, int k,
                                                                 int H, int Mpad, const int32_t *__restrict__ offsets,
                                                                 const int32_t *__restrict__ pad_off, int E,
                                                                 uint8_t *__restrict__ codes_t, uint8_t *__restrict__ sf_t,
                                                                 SfLayout Lt, RowCodes rows, float *__restrict__ g_part) {
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) uint8_t qc_smem[];
  uint16_t *ring = reinterpret_cast<uint16_t *>(qc_smem);  // [kDyRing][dy tile | Y tile]
  uint8_t *otile = qc_smem + kDyRing * 2 * kQcTileElems * 2;
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
  auto dy_ptr = [&](int r) -> const uint16_t * {
    return r < nvalid ? dy + static_cast<size_t>(s_tok[r]) * H : nullptr;
  };
  auto y_ptr = [&](int r) -> const uint16_t * { return r < nvalid ? Y + static_cast<size_t>(row0 + r) * H : nullptr; };
  const int first = blockIdx.y * kQcCols, step = gridDim.y * kQcCols;
  const int nt = first < H ? (H - first + step - 1) / step : 0;
  auto issue = [&](int i) {
    uint16_t *slot = ring + (i % kDyRing) * 2 * kQcTileElems;
    qc_issue(slot, first + i * step, dy_ptr, false);
    qc_issue(slot + kQcTileElems, first + i * step, y_ptr, true);  // one group per tile: both sources
  };
  const int r = threadIdx.x >> 1, bb = threadIdx.x & 1;  // row pass: row, 32-column block
  const size_t row_sf = atom_row(prow0 + r, H, rows.L);  // its scale bytes' row
  float gpart = 0.f;
  for (int i = 0; i < kDyRing - 1 && i < nt; ++i) issue(i);
  for (int it = 0; it < nt; ++it) {
    const int ahead = it + kDyRing - 1;
    if (ahead < nt) issue(ahead);
    cp_async_wait_pending(min(nt - 1, ahead) - it);  // this tile's group has landed
    __syncthreads();
    const uint16_t *tile = ring + (it % kDyRing) * 2 * kQcTileElems, *ytile = tile + kQcTileElems;
    const int c0 = first + it * step;
    {
      float v[32], yv[32];
      qc_row32(tile, r, bb, v);
      qc_row32(ytile, r, bb, yv);
#pragma unroll
      for (int i = 0; i < 32; ++i) gpart = fmaf(v[i], yv[i], gpart);
      const int prow = prow0 + r, kb = (c0 >> 5) + bb;
      rows.sf[row_sf + atom_kblock(kb)] =
          quant32(v, reinterpret_cast<uint4 *>(rows.codes + static_cast<size_t>(prow) * H + c0 + 32 * bb));
    }
    const int cc = threadIdx.x % kQcCols, b = threadIdx.x / kQcCols;  // 4 blocks of 32 tokens
    float v[32];
    qc_col32(tile, cc, b, v);
    sf_t[atom_row<kMxBN>(c0 + cc, Mpad, Lt) + atom_kblock((prow0 >> 5) + b)] =
        quant32(v, reinterpret_cast<uint4 *>(otile + cc * kQcOutStride + 32 * b));
    __syncthreads();
#pragma unroll
    for (int j = 0; j < (kQcCols * kQcRows / 16) / kQcThreads; ++j) {
      const int i = threadIdx.x + j * kQcThreads;
      const int orow = i >> 3, part = i & 7;  // output row (column c0 + orow), 16-byte piece
      *reinterpret_cast<uint4 *>(codes_t + static_cast<size_t>(c0 + orow) * Mpad + prow0 + part * 16) =
          *reinterpret_cast<const uint4 *>(otile + orow * kQcOutStride + part * 16);
    }
    __syncthreads();  // the tile's slot and the output tile are reused
  }
  gpart += __shfl_xor_sync(0xffffffffu, gpart, 1);  // the row's two 32-column halves
  if (bb == 0 && r < nvalid) g_part[static_cast<size_t>(row0 + r) * gridDim.y + blockIdx.y] = gpart;
}

// Weights quantised along their middle axis (the mxfp8 forward GEMMs' K),
// written transposed: W [E, R, C] bf16 (R the reduction axis, R % 128 == 0)
// -> codes [rows, R] with output row (e, c) = e * C + c (W_down: the down
// GEMM's B rows), or, interleaved for gate|up tiles, e * 2C + (c / 32) * 64 +
// half * 32 + c % 32 (W_gate half 0, W_up half 1: every 64 B rows hold 32
// gate columns then the same 32 up columns).  Optionally the same staged tile
// is also quantised along C, row by row (the backward GEMMs' weight operand,
// codes [E * R, C]), so each weight is read once for both.  Same staging and
// column walk as the token-axis quantiser.
__global__ void __launch_bounds__(kQcThreads, 3) quant_wT_kernel(const uint16_t *__restrict__ src, int R,
                                                                 int C, int interleave, int half,
                                                                 uint8_t *__restrict__ codes,
                                                                 uint8_t *__restrict__ sf, SfLayout L,
                                                                 RowCodes rows) {
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) uint8_t qc_smem[];
  uint16_t *ring = reinterpret_cast<uint16_t *>(qc_smem);
  uint8_t *otile = qc_smem + kQcRing * kQcTileElems * 2;
  const int grow0 = blockIdx.x * kQcRows;  // first source row (of E * R)
  const int e = grow0 / R, r0 = grow0 - e * R;
  auto out_row = [&](int c) {
    return interleave ? e * 2 * C + (c >> 5) * 64 + half * 32 + (c & 31) : e * C + c;
  };
  auto row_ptr = [&](int r) -> const uint16_t * { return src + static_cast<size_t>(grow0 + r) * C; };
  qc_walk(ring, blockIdx.y * kQcCols, gridDim.y * kQcCols, C, row_ptr, [&](const uint16_t *tile, int c0) {
    if (rows.codes) {  // along C: thread = (row, 32-column block)
      const int r = threadIdx.x >> 1, bb = threadIdx.x & 1;
      float v[32];
      qc_row32(tile, r, bb, v);
      const int grow = grow0 + r;
      rows.sf[atom_byte(grow, (c0 >> 5) + bb, C, rows.L)] =
          quant32(v, reinterpret_cast<uint4 *>(rows.codes + static_cast<size_t>(grow) * C + c0 + 32 * bb));
    }
    const int cc = threadIdx.x % kQcCols, b = threadIdx.x / kQcCols;  // 4 blocks of 32 rows
    float v[32];
    qc_col32(tile, cc, b, v);
    sf[atom_byte(out_row(c0 + cc), (r0 >> 5) + b, R, L)] =
        quant32(v, reinterpret_cast<uint4 *>(otile + cc * kQcOutStride + 32 * b));
    __syncthreads();
#pragma unroll
    for (int j = 0; j < (kQcCols * kQcRows / 16) / kQcThreads; ++j) {
      const int i = threadIdx.x + j * kQcThreads;
      const int r = i >> 3, part = i & 7;  // output row (column c0 + r), 16-byte piece
      *reinterpret_cast<uint4 *>(codes + static_cast<size_t>(out_row(c0 + r)) * R + r0 + part * 16) =
          *reinterpret_cast<const uint4 *>(otile + r * kQcOutStride + part * 16);
    }
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
                              RowCodes rows, cudaStream_t s, const int32_t *slot_of_row, int k, uint16_t *xp) {
  const int col_blocks = C / kQcCols < 4 ? C / kQcCols : 4;  // each loops over C / (64 * 4) column tiles
  const dim3 grid(static_cast<unsigned>(Mpad / kQcRows), static_cast<unsigned>(col_blocks));
  static DeviceOnce once;  // dynamic shared memory above 48 KB, opted in once per device
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(quant_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQcSmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(quant_cols_kernel, grid, dim3(kQcThreads), kQcSmem, s, 1, src, C, Mpad, offsets, pad_off, E,
                    codes, sf, L, rows, slot_of_row, k, xp);
}

cudaError_t launch_dy_quant(const uint16_t *dy, const uint16_t *Y, const int32_t *slot_of_row, int k, int H,
                            int Mpad, const int32_t *offsets, const int32_t *pad_off, int E, uint8_t *codes_t,
                            uint8_t *sf_t, SfLayout Lt, RowCodes rows, float *g_part, int col_blocks,
                            cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(Mpad / kQcRows), static_cast<unsigned>(col_blocks));
  static DeviceOnce once;  // dynamic shared memory above 48 KB, opted in once per device
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(dy_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDySmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(dy_quant_kernel, grid, dim3(kQcThreads), kDySmem, s, 1, dy, Y, slot_of_row, k, H, Mpad, offsets,
                    pad_off, E, codes_t, sf_t, Lt, rows, g_part);
}

int dy_quant_col_blocks(int H) { return H / kQcCols < 4 ? H / kQcCols : 4; }

cudaError_t launch_quant_wT(const uint16_t *W, int E, int R, int C, int interleave, int half,
                            uint8_t *codes, uint8_t *sf, SfLayout L, RowCodes rows, cudaStream_t s) {
  const int col_blocks = C / kQcCols < 4 ? C / kQcCols : 4;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(E) * R / kQcRows), static_cast<unsigned>(col_blocks));
  static DeviceOnce once;
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(quant_wT_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQcSmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(quant_wT_kernel, grid, dim3(kQcThreads), kQcSmem, s, 1, W, R, C, interleave, half, codes, sf, L,
                    rows);
}

}  // namespace moe
