// ffn_b1_i8.cu -- single-token gate-first sparse FFN with weight-only int8 or
// int4 weights (standard gate), streaming form; the per-row quantiser and the
// int4 packing.
//
// "Model Casting and Low-Parameter Gating", appendix Table 17, quantises the
// cast models weight-only to int8.  Convention of this library (the pages give
// none): symmetric, one fp32 scale per output channel -- per row of W1 and W3
// (unit i), per row of W2 (output element m) -- s = max|w| / 127, code =
// round-half-to-even(w / s) clamped to [-127, 127], decided in binary32.  The
// forward is the formula of "Model casting: compute the gate, then skip most of
// the FFN" with every weight replaced by q * s:
//     z_i = s1_i (q1[i, :] . x),   u_i = s3_i (q3[i, :] . x),   h_i = A(z_i) u_i
//     y_m = s2_m sum_{i live} q2t[i, m] h_i      (q2t = the codes of W2, transposed)
// Each block multiplies its partial y by s2 (staged in shared memory before the
// dependency wait) before adding it to the accumulator.  x and y are bf16.
//
// GB300 mapping: the pipeline of the bf16 streaming kernel (ffn_b1_stream.cu)
// with rows of D bytes instead of 2D -- the gate, which is always read in
// full, moves half the bytes.  A 16-byte chunk holds 16 codes, which pair with
// 16 values of x, widened to fp32 once per block in shared memory.  Codes are
// widened to fp32 exactly with a byte permute and a packed add (no int->float
// conversion instruction): the biased byte q + 128 becomes the low mantissa
// byte of 2^23.  q * x is exact in fp32 (7 x 8 significant bits); the sums
// are fp32, two lanes per packed fp32x2 FMA.
//
// int4 (same appendix, 7 in place of 127, and for W1 and W3 one scale per group
// of 64 consecutive columns instead of one per row -- with one int4 scale per
// row a single large entry rounds the rest of the row to zero): a row holds
// D / 2 bytes, byte b carrying codes 2b (low nibble) and 2b + 1 (high nibble) in
// two's complement.  A piece's dot product is scaled by its group's scale before
// it joins the lane's sum.  The kernel is the int8 one with 8-byte pieces of 16 codes in
// place of 16-byte pieces of 16 codes, so every piece still pairs with the same
// 16 values of x and the same 16 outputs: the lane and warp mappings, the staged
// x layout and the gathers are shared.  A nibble is widened like a byte: its sign
// bit flipped (code + 8), placed in the low mantissa bits of 2^23, 2^23 + 8
// subtracted.  There are no spin-waits in this file.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int QW = 12;        // warps per block (two blocks fit an SM)
constexpr int QT = QW * 32;
constexpr int QPIECE = 5;     // 16-byte chunks per lane per piece of a streamed gate row
constexpr int G4 = 64;        // int4: columns per scale group of W1 and W3 (four pieces of 16 codes)

__host__ __device__ constexpr size_t a16(size_t v) { return (v + 15) & ~size_t(15); }

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 lds_piece(const uint4* p) { return lds16(p); }
__device__ __forceinline__ uint2 lds_piece(const uint2* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
  return v;
}

// The piece of a code row that pairs with 16 values of x: 16 bytes of int8
// codes or 8 bytes of int4 codes.
template <int BITS> struct Piece;
template <> struct Piece<8> { using type = uint4; };
template <> struct Piece<4> { using type = uint2; };

__device__ __forceinline__ void cpa16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void pf_l2(const void* row, uint32_t bytes, int j, int nl) {
  const char* b = static_cast<const char*>(row);
  for (uint32_t off = (uint32_t)j * 128u; off < bytes; off += (uint32_t)nl * 128u)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(b + off));
}

// 4 int8 codes (one 32-bit word) -> 4 exact fp32 values, as 2 pairs.
__device__ __forceinline__ void widen_i8x4(uint32_t word, float2& v01, float2& v23) {
  const uint32_t w = word ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.f, -8388736.f);
  v01 = fadd2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u)),
                          __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u))), bias);
  v23 = fadd2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542u)),
                          __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543u))), bias);
}

// 8 int4 codes (one 32-bit word, code j in bits 4j .. 4j + 3) -> 8 exact fp32
// values, v[k] = (code 2k, code 2k + 1).  The biased even and odd codes are split
// into the bytes of two words once (a mask, a shift and a mask); each code then
// takes one byte permute into the low byte of 2^23, as in widen_i8x4.
__device__ __forceinline__ void widen_i4x8(uint32_t word, float2 (&v)[4]) {
  const uint32_t w = word ^ 0x88888888u;
  const uint32_t even = w & 0x0F0F0F0Fu, odd = (w >> 4) & 0x0F0F0F0Fu;
  const float2 bias = make_float2(-8388616.f, -8388616.f);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    v[k] = fadd2(make_float2(__uint_as_float(__byte_perm(even, 0x4B000000u, 0x7540u + k)),
                             __uint_as_float(__byte_perm(odd, 0x4B000000u, 0x7540u + k))),
                 bias);
}

// acc += code chunk c . x[16c, 16c + 16), two lanes of fp32 per FMA.  x is
// staged as fp32 in the interleaved layout xq[k * ncw + c] = x[16c + 4k .. +4),
// so lanes reading consecutive chunks read consecutive 16-byte words.
__device__ __forceinline__ void dot_chunk(const uint2& w, const float4* xq, int ncw, int c, float2& acc) {
  const uint32_t words[2] = {w.x, w.y};
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // word h: codes 8h .. 8h + 7, x quarters 2h and 2h + 1
    float2 v[4];
    widen_i4x8(words[h], v);
    const float4 xa = lds_f4(xq + (2 * h) * ncw + c), xb = lds_f4(xq + (2 * h + 1) * ncw + c);
    ffma2(acc, v[0], make_float2(xa.x, xa.y));
    ffma2(acc, v[1], make_float2(xa.z, xa.w));
    ffma2(acc, v[2], make_float2(xb.x, xb.y));
    ffma2(acc, v[3], make_float2(xb.z, xb.w));
  }
}
__device__ __forceinline__ void dot_chunk(const uint4& w, const float4* xq, int ncw, int c, float2& acc) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 v01, v23;
    widen_i8x4(words[k], v01, v23);
    const float4 xv = lds_f4(xq + k * ncw + c);
    ffma2(acc, v01, make_float2(xv.x, xv.y));
    ffma2(acc, v23, make_float2(xv.z, xv.w));
  }
}

// y partial += h * (the 16 codes of piece wv), outputs yr[0..16)
__device__ __forceinline__ void fold_piece(const uint4& wv, float h, float (&yr)[16]) {
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
  const float2 hh = make_float2(h, h);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 v01, v23;
    widen_i8x4(words[k], v01, v23);
    float2 a = make_float2(yr[4 * k], yr[4 * k + 1]), b = make_float2(yr[4 * k + 2], yr[4 * k + 3]);
    ffma2(a, v01, hh);
    ffma2(b, v23, hh);
    yr[4 * k] = a.x;
    yr[4 * k + 1] = a.y;
    yr[4 * k + 2] = b.x;
    yr[4 * k + 3] = b.y;
  }
}
__device__ __forceinline__ void fold_piece(const uint2& wv, float h, float (&yr)[16]) {
  const uint32_t words[2] = {wv.x, wv.y};
  const float2 hh = make_float2(h, h);
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    float2 v[4];
    widen_i4x8(words[w], v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 a = make_float2(yr[8 * w + 2 * k], yr[8 * w + 2 * k + 1]);
      ffma2(a, v[k], hh);
      yr[8 * w + 2 * k] = a.x;
      yr[8 * w + 2 * k + 1] = a.y;
    }
  }
}

__device__ __forceinline__ float lds_f32(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_u32(p)));
  return v;
}

// acc += piece c . x, scaled for int4 by the scale of the piece's group (gs: the row's
// group scales in shared memory); int8 rows are scaled once, after the sum.
template <int BITS, typename CT>
__device__ __forceinline__ void dot_piece(const CT& w, const float4* xq, int ncw, int c, float2& acc,
                                          const float* gs) {
  if constexpr (BITS == 4) {
    float2 part = make_float2(0.f, 0.f);
    dot_chunk(w, xq, ncw, c, part);
    const float sc = lds_f32(gs + (c >> 2));
    ffma2(acc, part, make_float2(sc, sc));
  } else {
    dot_chunk(w, xq, ncw, c, acc);
  }
}

template <typename CT>
__device__ __forceinline__ CT zero_piece();
template <>
__device__ __forceinline__ uint4 zero_piece<uint4>() { return make_uint4(0, 0, 0, 0); }
template <>
__device__ __forceinline__ uint2 zero_piece<uint2>() { return make_uint2(0, 0); }

template <typename CT>
__device__ __forceinline__ void load_piece_i8(CT (&w)[QPIECE], const CT* row, int pc, int lane, int ncw) {
#pragma unroll
  for (int k = 0; k < QPIECE; ++k) {
    const int c = pc * 32 * QPIECE + lane + 32 * k;
    w[k] = (c < ncw) ? ldg_stream(row + c) : zero_piece<CT>();
  }
}

template <int BITS, bool LOWRANK>
__global__ void __launch_bounds__(QT, 2) ffn_b1_i8_kernel(const B1Params p) {
  using CT = typename Piece<BITS>::type;
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int nch = D / 8;    // 16-byte bf16 chunks of x
  const int ncw = D / 16;   // pieces of 16 codes in a weight row (16 bytes int8, 8 bytes int4)
  const uint32_t row_bytes = (uint32_t)(D * BITS / 8);
  const int rq = (int)(row_bytes / 16);  // 16-byte units of a row (D % 64 == 0 for int4)
  const int ng = BITS == 4 ? D / G4 : 1;  // scales per row of W1 and of W3
  // the gate: rows of W1 over x, or (low-rank gate, int8) rows of U over t = V x, gcw pieces a row
  constexpr bool lowrank = LOWRANK;  // p.t holds t
  const int gcw = lowrank ? p.gate_k / 16 : ncw;              // the standard gate's rows are W1's
  const int rqg = lowrank ? p.gate_k * BITS / 8 / 16 : rq;    // 16-byte units of a gate row
  const int npg = (gcw + 32 * QPIECE - 1) / (32 * QPIECE);
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int cap = p.rows_cap;
  // shared: x | W2 scales | the block's W1, W3 scales | live list (unit, A(z), h) | counters |
  // live flags | prefetch / gather area
  uint8_t* sp = smem;
  float4* xq = reinterpret_cast<float4*>(sp);  // x widened to fp32 once per block (interleaved)
  sp += a16((size_t)D * 4);
  float4* gq = xq;  // the gate's vector in the same layout: x, or t for the low-rank gate
  if (lowrank) {
    gq = reinterpret_cast<float4*>(sp);
    sp += a16((size_t)p.gate_k * 4);
  }
  float* s2s = reinterpret_cast<float*>(sp);
  sp += a16((size_t)D * 4);
  float* s1s = reinterpret_cast<float*>(sp);  // [cap][ng] scales of the block's W1 rows, then of its W3 rows
  float* s3s = s1s + (size_t)cap * ng;
  sp += a16((size_t)cap * ng * 8);
  int* l_unit = reinterpret_cast<int*>(sp);
  float* l_a = reinterpret_cast<float*>(l_unit + cap);
  float* l_h = l_a + cap;
  int* misc = reinterpret_cast<int*>(l_h + cap);  // 0: live count
  uint8_t* l_mask = reinterpret_cast<uint8_t*>(misc + 4);
  sp += a16((size_t)cap * 13 + 16);
  uint4* srows = reinterpret_cast<uint4*>(sp);
  const CT* srow_p = reinterpret_cast<const CT*>(sp);  // the same area as rows of ncw pieces

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CT* G = static_cast<const CT*>(p.gate_w);
  const CT* W3 = static_cast<const CT*>(p.W3);
  const CT* W2t = static_cast<const CT*>(p.W2t);

  if (tid == 0) {
    pdl_launch_dependents();
    misc[0] = 0;
  }

  // Gate rows of the block: [0, R) copied into shared memory before the
  // dependency wait, [R, R + nreg) one per warp through registers (first two
  // pieces requested before the wait), the rest in shared-memory batches.
  const int nrows = row1 - row0;
  const int R = min(p.pref_rows, nrows);
  const int nreg = max(0, min(QW, nrows - R));
  auto copy_rows = [&](int first, int n) {
    const uint4* src = reinterpret_cast<const uint4*>(G + (size_t)(row0 + first) * gcw);
    for (int i = tid; i < n * rqg; i += QT) cpa16(srows + i, src + i);
    cpa_commit();
  };
  for (int i = tid; i < D / 4; i += QT) cpa16(s2s + 4 * i, p.s2 + 4 * i);  // committed with the rows
  for (int i = tid; i < (row1 - row0) * ng; i += QT) {  // scales of the block's units (weights: before the wait)
    s1s[i] = __ldg(p.s1 + (size_t)row0 * ng + i);
    s3s[i] = __ldg(p.s3 + (size_t)row0 * ng + i);
  }
  copy_rows(0, R);
  const int n_seq = warp < nreg ? npg : 0;
  const CT* my_row = G + (size_t)(row0 + R + warp) * gcw;
  CT wa[QPIECE], wb[QPIECE];
  if (n_seq > 0) load_piece_i8(wa, my_row, 0, lane, gcw);
  if (n_seq > 1) load_piece_i8(wb, my_row, 1, lane, gcw);
  if (tid == 0) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.x), "r"((uint32_t)nch * 16u)
                             : "memory");

  pdl_wait();  // x, the accumulators and the counters follow stream order
  for (int i = tid; i < nch; i += QT) {  // bf16 chunk i = float4 words 2i, 2i + 1 of x
    float v[8];
    Elt<bf16_tag>::unpack(__ldcg(static_cast<const uint4*>(p.x) + i), v);
    const int f0 = 2 * i, f1 = 2 * i + 1;  // word f: chunk f / 4, quarter f % 4
    xq[(f0 & 3) * ncw + (f0 >> 2)] = make_float4(v[0], v[1], v[2], v[3]);
    xq[(f1 & 3) * ncw + (f1 >> 2)] = make_float4(v[4], v[5], v[6], v[7]);
  }
  if (lowrank)  // t [r] fp32 from the t kernel: word f = t[4f .. 4f + 4), piece f / 4, quarter f % 4
    for (int f = tid; f < p.gate_k / 4; f += QT)
      gq[(f & 3) * gcw + (f >> 2)] = __ldcg(reinterpret_cast<const float4*>(p.t) + f);
  cpa_wait();
  __syncthreads();

  auto decide = [&](int q, float dotv) {  // dotv identical in every lane of the warp
    const float z = BITS == 4 ? dotv : s1s[q - row0] * dotv;  // int4: scaled per group already
    const float a = activation(p.act, z);
    const bool live = is_live(a, p.thr);
    if (lane == 0) {
      l_mask[q - row0] = live ? 1 : 0;
      if (live) {
        const int j = atomicAdd(misc, 1);
        l_unit[j] = q;
        l_a[j] = a;
      }
    }
    if (live) {
      pf_l2(W3 + (size_t)q * ncw, row_bytes, lane, 32);
      pf_l2(W2t + (size_t)q * ncw, row_bytes, lane, 32);
    }
  };
  auto shared_rows = [&](int first, int n) {
    for (int i = warp; i < n; i += QW) {
      const CT* r = srow_p + (size_t)i * gcw;
      const float* gs = s1s + (size_t)(first + i) * ng;
      float2 acc = make_float2(0.f, 0.f);
      for (int c = lane; c < gcw; c += 32) dot_piece<BITS>(lds_piece(r + c), gq, gcw, c, acc, gs);
      decide(row0 + first + i, warp_sum(acc.x + acc.y));
    }
  };
  shared_rows(0, R);
  __syncthreads();
  int next = R + nreg;
  int nb1 = min(R, nrows - next);
  if (nb1 > 0) copy_rows(next, nb1);

  float2 acc = make_float2(0.f, 0.f);
  const float* my_gs = s1s + (size_t)(R + warp) * ng;
  auto consume = [&](const CT(&w)[QPIECE], int pc) {
#pragma unroll
    for (int k = 0; k < QPIECE; ++k) {
      const int c = pc * 32 * QPIECE + lane + 32 * k;
      if (c < gcw) dot_piece<BITS>(w[k], gq, gcw, c, acc, my_gs);
    }
    if (pc == npg - 1) {
      const float d = warp_sum(acc.x + acc.y);
      acc = make_float2(0.f, 0.f);
      decide(row0 + R + warp, d);
    }
  };
  for (int pc = 0; pc < n_seq; pc += 2) {
    consume(wa, pc);
    if (pc + 2 < n_seq) load_piece_i8(wa, my_row, pc + 2, lane, gcw);
    if (pc + 1 < n_seq) {
      consume(wb, pc + 1);
      if (pc + 3 < n_seq) load_piece_i8(wb, my_row, pc + 3, lane, gcw);
    }
  }
  while (nb1 > 0) {
    cpa_wait();
    __syncthreads();
    shared_rows(next, nb1);
    __syncthreads();
    next += nb1;
    nb1 = min(R, nrows - next);
    if (nb1 > 0) copy_rows(next, nb1);
  }
  __syncthreads();
  const int n_live = misc[0];

  // ---- gathers.  Warp w owns code chunks [cs0, cs0 + cs_n) of a W2^T row,
  // i.e. outputs [16 cs0, 16 (cs0 + cs_n)); lane l holds the 16 outputs of
  // chunk cs0 + l (and of cs0 + 32 + l in a second pass for wide rows).
  const int per = (ncw + QW - 1) / QW;
  const int cs0 = warp * per;
  const int cs_n = min(per, ncw - cs0);
  const bool owns = lane < cs_n;
  const CT* col = W2t + cs0 + lane;
  const int RB = p.gather_rows;
  const bool dbl = (p.flags & FLAG_DOUBLE_ACT) != 0;
  float yr[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) yr[v] = 0.f;
  auto fold = [&](const CT& wv, float h) { fold_piece(wv, h, yr); };
  CT r8[8];
  for (int b0 = 0; b0 < n_live; b0 += RB) {
    const int nb = min(RB, n_live - b0);
    for (int i = tid; i < nb * rq; i += QT) {
      const int u = i / rq, c = i - u * rq;
      cpa16(srows + i, reinterpret_cast<const uint4*>(W3 + (size_t)l_unit[b0 + u] * ncw) + c);
    }
    cpa_commit();
#pragma unroll
    for (int m = 0; m < 8; ++m)
      r8[m] = (owns && m < nb) ? ldg_stream(col + (size_t)l_unit[b0 + m] * ncw) : zero_piece<CT>();
    cpa_wait();
    __syncthreads();
    for (int u = warp; u < nb; u += QW) {
      const CT* r = srow_p + (size_t)u * ncw;
      const int ur = l_unit[b0 + u] - row0;
      float2 acc2 = make_float2(0.f, 0.f);
      for (int c = lane; c < ncw; c += 32) dot_piece<BITS>(lds_piece(r + c), xq, ncw, c, acc2, s3s + (size_t)ur * ng);
      const float uval = BITS == 4 ? warp_sum(acc2.x + acc2.y) : s3s[ur] * warp_sum(acc2.x + acc2.y);
      if (lane == 0) l_h[b0 + u] = l_a[b0 + u] * (dbl ? activation(p.act, uval) : uval);
    }
    __syncthreads();
    if (owns) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < nb) fold(r8[m], l_h[b0 + m]);
      for (int j = 8; j < nb; j += 4) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
          r8[m] = j + m < nb ? ldg_stream(col + (size_t)l_unit[b0 + j + m] * ncw) : zero_piece<CT>();
#pragma unroll
        for (int m = 0; m < 4; ++m)
          if (j + m < nb) fold(r8[m], l_h[b0 + j + m]);
      }
    }
    __syncthreads();
  }
  float* yc = p.yacc + (size_t)(blockIdx.x % YACC_COPIES) * D;
  auto add_scaled = [&](int chunk) {  // y[16 chunk + v] += s2[16 chunk + v] * yr[v]
    const float4* sc = reinterpret_cast<const float4*>(s2s + (size_t)chunk * 16);
#pragma unroll
    for (int v = 0; v < 16; v += 4) {
      const float4 f = sc[v / 4];
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)chunk * 16 + v),
                make_float4(f.x * yr[v], f.y * yr[v + 1], f.z * yr[v + 2], f.w * yr[v + 3]));
    }
  };
  if (n_live > 0 && owns) add_scaled(cs0 + lane);
  if (n_live > 0 && lane + 32 < cs_n) {  // rows wider than 32 chunks per warp
#pragma unroll
    for (int v = 0; v < 16; ++v) yr[v] = 0.f;
    for (int j = 0; j < n_live; j += 4) {
#pragma unroll
      for (int m = 0; m < 4; ++m)
        r8[m] = j + m < n_live ? ldg_stream(col + 32 + (size_t)l_unit[j + m] * ncw) : zero_piece<CT>();
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (j + m < n_live) fold(r8[m], l_h[j + m]);
    }
    add_scaled(cs0 + 32 + lane);
  }
  if (tid == 0 && n_live > 0) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot, n_live);
  if (p.mask)
    for (int i = tid; i < nrows; i += QT) p.mask[row0 + i] = l_mask[i];
}

// One block per row of a bf16 matrix: s = max|w| / QMAX, codes = round-half-even(w / s)
// clamped to [-QMAX, QMAX] (binary32 division, correctly rounded); s = 0 and codes 0 for
// an all-zero row.  QMAX = 127 (int8) or 7 (int4, one code per byte before packing).
template <int QMAX>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ src,
                                                            int8_t* __restrict__ dst, float* __restrict__ scale,
                                                            int cols) {
  __shared__ float red[8];
  const uint16_t* w = src + (size_t)blockIdx.x * cols;
  int8_t* q = dst + (size_t)blockIdx.x * cols;
  float amax = 0.f;
  for (int j = threadIdx.x; j < cols; j += 256) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)w[j] << 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) amax = fmaxf(amax, red[k]);
  const float s = __fdiv_rn(amax, (float)QMAX);
  if (threadIdx.x == 0) scale[blockIdx.x] = s;
  for (int j = threadIdx.x; j < cols; j += 256) {
    int v = 0;
    if (s > 0.f) {
      v = __float2int_rn(__fdiv_rn(__uint_as_float((uint32_t)w[j] << 16), s));
      v = max(-QMAX, min(QMAX, v));
    }
    q[j] = (int8_t)v;
  }
}

// One block per row of a bf16 matrix, one scale per group of G4 columns (int4 W1, W3):
// s[row * (cols / G4) + g] = max|w over the group| / 7, codes as quantize_rows_kernel<7>.
// A warp takes a group, two columns per lane.
__global__ void __launch_bounds__(256) quantize_groups4_kernel(const uint16_t* __restrict__ src,
                                                               int8_t* __restrict__ dst, float* __restrict__ scale,
                                                               int cols) {
  const int lane = threadIdx.x & 31, ng = cols / G4;
  const uint16_t* w = src + (size_t)blockIdx.x * cols;
  int8_t* q = dst + (size_t)blockIdx.x * cols;
  for (int g = threadIdx.x >> 5; g < ng; g += 8) {
    const float a = __uint_as_float((uint32_t)w[g * G4 + lane] << 16);
    const float b = __uint_as_float((uint32_t)w[g * G4 + 32 + lane] << 16);
    float amax = fmaxf(fabsf(a), fabsf(b));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 7.f);
    if (lane == 0) scale[(size_t)blockIdx.x * ng + g] = s;
    int va = 0, vb = 0;
    if (s > 0.f) {
      va = max(-7, min(7, __float2int_rn(__fdiv_rn(a, s))));
      vb = max(-7, min(7, __float2int_rn(__fdiv_rn(b, s))));
    }
    q[g * G4 + lane] = (int8_t)va;
    q[g * G4 + 32 + lane] = (int8_t)vb;
  }
}

// Low-rank gate with int8 weights: t_k = sV_k (qV[k, :] . x), one warp per row of V (D % 16 == 0),
// the row's 16-byte pieces requested before the dependency wait, x read from L2 after it.
constexpr int TW = 8;  // warps (rows of V) per block
__global__ void __launch_bounds__(TW * 32) lopa_t_i8_kernel(const int8_t* __restrict__ qV, const float* __restrict__ sV,
                                                            const uint16_t* __restrict__ x, float* __restrict__ t,
                                                            int r, int D) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, k = blockIdx.x * TW + warp;
  const int npc = D / 16;
  const uint4* row = reinterpret_cast<const uint4*>(qV + (size_t)min(k, r - 1) * D);
  constexpr int PL = 8;  // pieces held per lane (D <= 4096)
  uint4 w[PL];
#pragma unroll
  for (int j = 0; j < PL; ++j) w[j] = (lane + 32 * j < npc && k < r) ? ldg_stream(row + lane + 32 * j) : make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();  // x follows stream order
  // every x piece requested at once: one L2 round trip, not one per piece
  uint4 xr[PL][2];
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    const int c = lane + 32 * j;
    const uint4* xp = reinterpret_cast<const uint4*>(x) + 2 * c;
    xr[j][0] = c < npc ? __ldcg(xp) : make_uint4(0, 0, 0, 0);
    xr[j][1] = c < npc ? __ldcg(xp + 1) : make_uint4(0, 0, 0, 0);
  }
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    const int c = lane + 32 * j;
    if (c >= npc) break;
    float xa[8], xb[8];
    Elt<bf16_tag>::unpack(xr[j][0], xa);
    Elt<bf16_tag>::unpack(xr[j][1], xb);
    const float xv[16] = {xa[0], xa[1], xa[2], xa[3], xa[4], xa[5], xa[6], xa[7],
                          xb[0], xb[1], xb[2], xb[3], xb[4], xb[5], xb[6], xb[7]};
    const uint32_t words[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float2 v01, v23;
      widen_i8x4(words[q], v01, v23);
      ffma2(acc, v01, make_float2(xv[4 * q], xv[4 * q + 1]));
      ffma2(acc, v23, make_float2(xv[4 * q + 2], xv[4 * q + 3]));
    }
  }
  const float d = warp_sum(acc.x + acc.y);
  if (lane == 0 && k < r) t[k] = sV[k] * d;
}

// int4 codes, one per byte in [-7, 7] -> two per byte (code 2i in the low nibble); a code
// outside that range sets DEV_ERR_CHECK in *err and packs as 0.
__global__ void pack_int4_kernel(const int8_t* __restrict__ codes, uint8_t* __restrict__ out, size_t n_bytes,
                                 int* err) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_bytes; i += (size_t)gridDim.x * blockDim.x) {
    int lo = codes[2 * i], hi = codes[2 * i + 1];
    if (lo < -7 || lo > 7 || hi < -7 || hi > 7) {
      atomicOr(err, DEV_ERR_CHECK);
      lo = (lo < -7 || lo > 7) ? 0 : lo;
      hi = (hi < -7 || hi > 7) ? 0 : hi;
    }
    out[i] = (uint8_t)((lo & 0xF) | ((hi & 0xF) << 4));
  }
}

// two int4 codes per byte -> one code per byte (sign-extended)
__global__ void unpack_int4_kernel(const uint8_t* __restrict__ in, int8_t* __restrict__ codes, size_t n_bytes) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_bytes; i += (size_t)gridDim.x * blockDim.x) {
    const int b = in[i];
    codes[2 * i] = (int8_t)(((b & 0xF) ^ 8) - 8);
    codes[2 * i + 1] = (int8_t)(((b >> 4) ^ 8) - 8);
  }
}

}  // namespace

StreamPlan plan_ffn_b1_i8(int D, int gate_k, int rows_cap, int bits, bool lowrank) {
  StreamPlan pl;
  const size_t row = (size_t)D * bits / 8;        // bytes of a gathered W3 code row
  const size_t grow = (size_t)gate_k * bits / 8;  // bytes of a gate code row (W1, or U of the low-rank gate)
  const size_t ng = bits == 4 ? (size_t)(D / G4) : 1;  // W1 and W3 scales per row
  // two blocks per SM (the next call's blocks prefetch while this call runs):
  // at most 110 KB per block, of which the gate-row area takes what is left
  const size_t tq = lowrank ? a16((size_t)gate_k * 4) : 0;  // the staged t of the low-rank gate
  const size_t fixed = 2 * a16((size_t)D * 4) + tq + a16((size_t)rows_cap * ng * 8) + a16((size_t)rows_cap * 13 + 16);
  const size_t budget = 110u * 1024u;
  const size_t free_area = budget > fixed ? budget - fixed : 0;
  pl.pref_rows = (int)std::min<size_t>((size_t)rows_cap, std::max<size_t>(1, free_area / grow));
  const size_t area = std::max((size_t)pl.pref_rows * grow, (size_t)std::min(rows_cap, 16) * row);
  pl.gather_rows = (int)std::max<size_t>(1, area / row);
  pl.smem = fixed + area;
  return pl;
}

cudaError_t ffn_b1_i8_prepare(size_t max_smem) {
  cudaError_t e = cudaSuccess;
  for (auto k : {ffn_b1_i8_kernel<8, false>, ffn_b1_i8_kernel<4, false>, ffn_b1_i8_kernel<8, true>}) {
    if (!e) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    if (!e) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  return e;
}

cudaError_t launch_ffn_b1_i8(const B1Params& p, int grid, size_t smem, cudaStream_t s, int bits) {
  if (p.t) {  // the low-rank gate: int8 only
    if (bits != 8) return cudaErrorInvalidValue;
    return launch_pdl(ffn_b1_i8_kernel<8, true>, dim3(grid), dim3(QT), smem, s, p);
  }
  return bits == 4 ? launch_pdl(ffn_b1_i8_kernel<4, false>, dim3(grid), dim3(QT), smem, s, p)
                   : launch_pdl(ffn_b1_i8_kernel<8, false>, dim3(grid), dim3(QT), smem, s, p);
}

cudaError_t launch_quantize_rows(const void* src_bf16, int8_t* dst, float* scale, int rows, int cols, cudaStream_t s,
                                 int qmax) {
  if (rows <= 0) return cudaSuccess;
  if (qmax == 7)
    quantize_rows_kernel<7><<<rows, 256, 0, s>>>(static_cast<const uint16_t*>(src_bf16), dst, scale, cols);
  else
    quantize_rows_kernel<127><<<rows, 256, 0, s>>>(static_cast<const uint16_t*>(src_bf16), dst, scale, cols);
  return cudaGetLastError();
}

cudaError_t launch_quantize_groups4(const void* src_bf16, int8_t* dst, float* scale, int rows, int cols,
                                    cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  quantize_groups4_kernel<<<rows, 256, 0, s>>>(static_cast<const uint16_t*>(src_bf16), dst, scale, cols);
  return cudaGetLastError();
}

cudaError_t launch_lopa_t_i8(const void* qV, const float* sV, const void* x, float* t, int r, int D, cudaStream_t s) {
  if (D % 16 || D > 32 * 8 * 16 || r < 1) return cudaErrorInvalidValue;
  return launch_pdl(lopa_t_i8_kernel, dim3((r + TW - 1) / TW), dim3(TW * 32), 0, s, static_cast<const int8_t*>(qV),
                    sV, static_cast<const uint16_t*>(x), t, r, D);
}

cudaError_t launch_pack_int4(const int8_t* codes, void* packed, size_t n_codes, int* err, cudaStream_t s) {
  if (n_codes == 0) return cudaSuccess;
  const size_t n = n_codes / 2;
  const int grid = (int)std::min<size_t>(4096, (n + 255) / 256);
  pack_int4_kernel<<<grid, 256, 0, s>>>(codes, static_cast<uint8_t*>(packed), n, err);
  return cudaGetLastError();
}

cudaError_t launch_unpack_int4(const void* packed, int8_t* codes, size_t n_codes, cudaStream_t s) {
  if (n_codes == 0) return cudaSuccess;
  const size_t n = n_codes / 2;
  const int grid = (int)std::min<size_t>(4096, (n + 255) / 256);
  unpack_int4_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(packed), codes, n);
  return cudaGetLastError();
}

}  // namespace sffn
