// epilogue.cuh -- epilogues of the grouped GEMMs: read one warp's 32 TMEM lanes
// of a 128 x 256 fp32 accumulator and write the layer's bf16 outputs (fused
// SwiGLU for the forward gate/up GEMM, fused dSwiGLU for dA).  Shared by the
// bf16 GEMM engine (gemm.cu) and the MXFP8 one (gemm_mx.cu).  `P` is any
// parameter struct with the fields used below (H, I, G, U, w_row, o0..o3).
#pragma once

#include "common.cuh"

namespace moe {

struct Tile {
  int e;        // expert
  int m0;       // first output row of the pair (ragged M: permuted row; ragged K: dW row)
  int row_end;  // ragged M: end of the expert's rows
  int n0;       // first output column
  int nkb;      // K blocks
  int krow0;    // ragged K: expert's first row
  int kcount;   // ragged K: expert's rows
};

__device__ __forceinline__ void store32_bf16(uint16_t *dst, const float (&v)[32]) {
  uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d[q] = w;
  }
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + __expf(-z)); }

// Epilogue of one tile for one warp (32 rows).  tb: TMEM address of this
// warp's lanes at the accumulator's first column.  NCH: 32-column chunks in
// the tile's unpaired accumulator (8 for 256 columns, 6 for 192).
template <int MODE, class P, int NCH = 8>
__device__ __forceinline__ void epilogue_tile(const Tile &t, uint32_t tb, int rit, const P &p) {
  uint32_t r0[32], r1[32];
  float v0[32], v1[32], v2[32];
  if constexpr (MODE == kFwdGateUp) {
    const int row = t.m0 + rit;
    const bool rv = row < t.row_end;
    const float w = rv ? __ldg(p.w_row + row) : 0.f;
    for (int c = 0; c < 4; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.I) break;
      tmem_ld32(tb + 32 * c, r0);
      tmem_ld32(tb + 128 + 32 * c, r1);
      tmem_ld_wait();
      if (rv) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float g = __uint_as_float(r0[i]), u = __uint_as_float(r1[i]);
          v0[i] = g * sigmoidf_(g) * u;  // SwiGLU
          v1[i] = g;
          v2[i] = u;
        }
        const size_t off = static_cast<size_t>(row) * p.I + col;
        store32_bf16(p.o0 + off, v0);
        store32_bf16(p.o1 + off, v1);
        store32_bf16(p.o2 + off, v2);
#pragma unroll
        for (int i = 0; i < 32; ++i) v0[i] *= w;  // A_w = w * A, the dW_down operand
        store32_bf16(p.o3 + off, v0);
      }
    }
  } else if constexpr (MODE == kFwdDown || MODE == kBwdDX) {
    const int row = t.m0 + rit;
    const bool rv = row < t.row_end;
    for (int c = 0; c < NCH; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.H) break;
      tmem_ld32(tb + 32 * c, r0);
      tmem_ld_wait();
      if (rv) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r0[i]);
        store32_bf16(p.o0 + static_cast<size_t>(row) * p.H + col, v0);
      }
    }
  } else if constexpr (MODE == kBwdDA) {
    const int row = t.m0 + rit;
    const bool rv = row < t.row_end;
    const float w = rv ? __ldg(p.w_row + row) : 0.f;  // dA = w * (dy . W_down^T)
    // G and U of the next 32-column chunk are loaded while this chunk is computed
    uint4 gq[4], uq[4], gn[4], un[4];
    const size_t rowoff = static_cast<size_t>(rv ? row : 0) * p.I;
    if (rv && t.n0 < p.I) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        gq[q] = __ldg(reinterpret_cast<const uint4 *>(p.G + rowoff + t.n0) + q);
        uq[q] = __ldg(reinterpret_cast<const uint4 *>(p.U + rowoff + t.n0) + q);
      }
    }
    for (int c = 0; c < NCH; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.I) break;
      const bool next = c + 1 < NCH && col + 32 < p.I;
      if (rv && next) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          gn[q] = __ldg(reinterpret_cast<const uint4 *>(p.G + rowoff + col + 32) + q);
          un[q] = __ldg(reinterpret_cast<const uint4 *>(p.U + rowoff + col + 32) + q);
        }
      }
      tmem_ld32(tb + 32 * c, r0);
      tmem_ld_wait();
      if (rv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t gw[4] = {gq[q].x, gq[q].y, gq[q].z, gq[q].w};
          const uint32_t uw[4] = {uq[q].x, uq[q].y, uq[q].z, uq[q].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            v1[8 * q + 2 * h] = bf16_lo(gw[h]);
            v1[8 * q + 2 * h + 1] = bf16_hi(gw[h]);
            v2[8 * q + 2 * h] = bf16_lo(uw[h]);
            v2[8 * q + 2 * h + 1] = bf16_hi(uw[h]);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float da = w * __uint_as_float(r0[i]), g = v1[i], u = v2[i];
          const float s = sigmoidf_(g);
          v0[i] = da * u * s * (1.f + g * (1.f - s));  // dG
          v1[i] = da * g * s;                          // dU = dA * silu(G)
        }
        store32_bf16(p.o0 + rowoff + col, v0);
        store32_bf16(p.o1 + rowoff + col, v1);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        gq[q] = gn[q];
        uq[q] = un[q];
      }
    }
  } else if constexpr (MODE == kBwdDWDown) {
    const int i_row = t.m0 + rit;
    const bool rv = i_row < p.I;
    for (int c = 0; c < NCH; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.H) break;
      if (t.nkb > 0) {
        tmem_ld32(tb + 32 * c, r0);
        tmem_ld_wait();
      }
      if (rv) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v0[i] = t.nkb > 0 ? __uint_as_float(r0[i]) : 0.f;
        store32_bf16(p.o0 + (static_cast<size_t>(t.e) * p.I + i_row) * p.H + col, v0);
      }
    }
  } else {  // kBwdDWGateUp
    const int h_row = t.m0 + rit;
    const bool rv = h_row < p.H;
    for (int c = 0; c < 4; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.I) break;
      if (t.nkb > 0) {
        tmem_ld32(tb + 32 * c, r0);
        tmem_ld32(tb + 128 + 32 * c, r1);
        tmem_ld_wait();
      }
      if (rv) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v0[i] = t.nkb > 0 ? __uint_as_float(r0[i]) : 0.f;
          v1[i] = t.nkb > 0 ? __uint_as_float(r1[i]) : 0.f;
        }
        const size_t off = (static_cast<size_t>(t.e) * p.H + h_row) * p.I + col;
        store32_bf16(p.o0 + off, v0);
        store32_bf16(p.o1 + off, v1);
      }
    }
  }
}

}  // namespace moe
