// rope.cuh -- the rotation angle of rotate-half RoPE on the device.
//
// SimSD section 3 "Position Encoding Alignment": a new token at position pos
// rotates element pair (d, d + hd/2) by pos * base^(-2d/hd).  Positions reach
// ~3.3e4, where a plain fp32 product is off by ~2e-3 rad, so the angle is
// formed as an unevaluated sum: the frequency as two floats hi + lo (from
// fp64 on the host), pos * hi with its exact rounding error recovered by an
// fma, then reduced modulo 2*pi with Cody and Waite's split constant (2*pi =
// C1 + C2, each product folded in by one fma) -- ~3e-7 rad, fp32 only (the
// GB300's fp64 rate is a small fraction of its fp32 rate).  Positions >= 2^24
// use fp64.  Sine and cosine of the reduced angle are fp32.
#pragma once

#include "internal.h"

namespace simsd {

// (cos, sin) of the angle of frequency d at position pos.
__device__ __forceinline__ float2 rope_cs(const RopeTable &tab, int d, int pos) {
  // 2*pi = C1 + C2 (C1 the float nearest 2*pi, C2 the float nearest the rest)
  const float C1 = 6.28318548202514648f, C2 = -1.7484555314695172e-07f;
  const float inv_two_pi = 0.159154943091895336f;
  float r;
  if (pos < (1 << 24)) {
    const float p = (float)pos;                       // exact
    const float t = p * tab.hi[d];
    const float t_lo = fmaf(p, tab.lo[d], fmaf(p, tab.hi[d], -t));  // rest of p*(hi+lo)
    const float n = rintf(t * inv_two_pi);
    r = fmaf(-n, C2, fmaf(-n, C1, t)) + t_lo;         // t + t_lo - 2*pi*n
  } else {
    const double two_pi = 6.283185307179586476925286766559;
    const double th = (double)pos * tab.inv_freq[d];
    r = (float)fma(-rint(th * (1.0 / two_pi)), two_pi, th);
  }
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(c, s);
}

}  // namespace simsd
