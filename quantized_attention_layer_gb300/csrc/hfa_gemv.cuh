// hfa_gemv.cuh -- the pieces of the dequantising Q8_0 GEMV shared by the persistent
// kernels (the attention step and the FFN step): tagged partial sums exchanged between
// CTAs without a grid barrier, the 16 x 32 tile times the split fp16 operand on the warp
// MMA, the operand's word order and its per-row power-of-two scale.
#pragma once
#include "hfa_common.cuh"

namespace hfa {

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// L2 loads the compiler keeps in place: never issued ahead of the branch that guards them
__device__ __forceinline__ unsigned long long ldcg_pinned64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
// Tagged partial sums: 8 bytes (f32 bits | step tag << 32) stored and loaded as one
// morally strong 64-bit access, so that a reader sees a value together with the step it
// belongs to and needs no fence or barrier to know that it is there.
__device__ __forceinline__ void st_tagged(unsigned long long* p, float v, uint32_t tag) {
  const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long* p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
// two adjacent entries (p 16-byte aligned), each read as one 64-bit relaxed access
__device__ __forceinline__ void ld_tagged2(const unsigned long long* p, unsigned long long& w0,
                                           unsigned long long& w1) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
}
__device__ __forceinline__ float tagged_value(unsigned long long w) {
  return __uint_as_float((uint32_t)w);
}
// One Q8_0 tile (16 rows x 32 columns) times every batch tile of the operand.
template <int NT>
__device__ __forceinline__ void q8_tile_mma(float (&acc)[NT][4], const uint4 w, uint32_t dbits,
                                            uint32_t xrow) {
  uint32_t A0[4], A1[4];
  A0[0] = u8x2_to_h2(w.x, kSelLo);
  A0[1] = u8x2_to_h2(w.y, kSelLo);
  A0[2] = u8x2_to_h2(w.x, kSelHi);
  A0[3] = u8x2_to_h2(w.y, kSelHi);
  A1[0] = u8x2_to_h2(w.z, kSelLo);
  A1[1] = u8x2_to_h2(w.w, kSelLo);
  A1[2] = u8x2_to_h2(w.z, kSelHi);
  A1[3] = u8x2_to_h2(w.w, kSelHi);
  const __half2 d2 = *reinterpret_cast<const __half2*>(&dbits);
  const float dg = __low2float(d2), dg8 = __high2float(d2);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4 xb = lds128(xrow + nt * 512);
    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16(tmp, A0, xb.x, xb.y);
    mma_f16(tmp, A1, xb.z, xb.w);
    acc[nt][0] = fmaf(tmp[0], dg, acc[nt][0]);
    acc[nt][1] = fmaf(tmp[1], dg, acc[nt][1]);
    acc[nt][2] = fmaf(tmp[2], dg8, acc[nt][2]);
    acc[nt][3] = fmaf(tmp[3], dg8, acc[nt][3]);
  }
}

// Two tiles at once: the same as two q8_tile_mma calls, with the two tiles' MMAs
// interleaved so that each one's latency hides behind the other's.
template <int NT>
__device__ __forceinline__ void q8_tile2_mma(float (&acc)[NT][4], const uint4 wa, uint32_t da,
                                             uint32_t xa, const uint4 wb, uint32_t db,
                                             uint32_t xb) {
  uint32_t A0[4], A1[4], B0[4], B1[4];
  A0[0] = u8x2_to_h2(wa.x, kSelLo);
  A0[1] = u8x2_to_h2(wa.y, kSelLo);
  A0[2] = u8x2_to_h2(wa.x, kSelHi);
  A0[3] = u8x2_to_h2(wa.y, kSelHi);
  A1[0] = u8x2_to_h2(wa.z, kSelLo);
  A1[1] = u8x2_to_h2(wa.w, kSelLo);
  A1[2] = u8x2_to_h2(wa.z, kSelHi);
  A1[3] = u8x2_to_h2(wa.w, kSelHi);
  B0[0] = u8x2_to_h2(wb.x, kSelLo);
  B0[1] = u8x2_to_h2(wb.y, kSelLo);
  B0[2] = u8x2_to_h2(wb.x, kSelHi);
  B0[3] = u8x2_to_h2(wb.y, kSelHi);
  B1[0] = u8x2_to_h2(wb.z, kSelLo);
  B1[1] = u8x2_to_h2(wb.w, kSelLo);
  B1[2] = u8x2_to_h2(wb.z, kSelHi);
  B1[3] = u8x2_to_h2(wb.w, kSelHi);
  const __half2 d2a = *reinterpret_cast<const __half2*>(&da);
  const __half2 d2b = *reinterpret_cast<const __half2*>(&db);
  const float ga = __low2float(d2a), ga8 = __high2float(d2a);
  const float gb = __low2float(d2b), gb8 = __high2float(d2b);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4 xva = lds128(xa + nt * 512), xvb = lds128(xb + nt * 512);
    float ta[4] = {0.f, 0.f, 0.f, 0.f}, tb[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16(ta, A0, xva.x, xva.y);
    mma_f16(tb, B0, xvb.x, xvb.y);
    mma_f16(ta, A1, xva.z, xva.w);
    mma_f16(tb, B1, xvb.z, xvb.w);
    acc[nt][0] = fmaf(ta[0], ga, acc[nt][0]);
    acc[nt][1] = fmaf(ta[1], ga, acc[nt][1]);
    acc[nt][2] = fmaf(ta[2], ga8, acc[nt][2]);
    acc[nt][3] = fmaf(ta[3], ga8, acc[nt][3]);
    acc[nt][0] = fmaf(tb[0], gb, acc[nt][0]);
    acc[nt][1] = fmaf(tb[1], gb, acc[nt][1]);
    acc[nt][2] = fmaf(tb[2], gb8, acc[nt][2]);
    acc[nt][3] = fmaf(tb[3], gb8, acc[nt][3]);
  }
}

// Operand word index of the column pair (cc, cc + 1) of batch row b: block cc / 32,
// k-step and half of the m16n8k16 B fragment; batch row b in the n8 tile b / 4, as
// column 2 (b % 4) (fp16 hi) and 2 (b % 4) + 1 (fp16 lo).  The lo word is 16 further.
template <int NT>
__device__ __forceinline__ int operand_word(int cc, int b) {
  const int jb = cc >> 5, w32 = cc & 31;
  const int ks = w32 >> 4, within = w32 & 15;
  const int hf = within >> 3, t = (within & 7) >> 1;
  const int nt = b >> 2, gh = 2 * (b & 3);
  return ((jb * NT + nt) * 32 + gh * 4 + t) * 4 + 2 * ks + hf;
}

// power-of-two scale that brings the largest |value| m of a row to [2^14, 2^15)
__device__ __forceinline__ int scale_exp(unsigned mbits) {
  if (mbits == 0u) return 0;
  int e = (int)((mbits >> 23) & 0xffu);
  if (e == 0) e = 1;  // subnormal
  int se = 141 - e;   // 14 - (e - 127)
  return se < -120 ? -120 : (se > 120 ? 120 : se);
}
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

}  // namespace hfa
