// rope_phase.cu -- the rotary angle as an exact fixed-point phase (host side).
//
// A rotary pair turns by theta = p * omega, omega = base^(-2i/d_axis), at the
// token's integer position p on the pair's axis. The time coordinate is the
// absolute latent-frame index of the stream (H3 project page, "Interactive
// Coding Worlds with Real-time Streaming Diffusion Render", section 3.2
// Iteration 4), which grows without bound, so p * omega cannot be rounded to
// a float: at p = 2^24 a float product is already off by a radian.
//
// The rotation needs theta modulo 2*pi only, that is the fractional part of
// p * c with c = omega / (2*pi) turns per position step. The host computes c
// once per pair as a 96-bit binary fraction C = round(c * 2^96); the kernels
// then form frac(p * c) with 64-bit integer arithmetic (sr::rope_angle in
// sr_kernels.h), exact up to the rounding of C, whose error of at most
// |p| * 2^-97 turns stays below 2^-55 turns for |p| < 2^42.
//
// C needs c to about 2^-100, beyond float64. It is computed in double-double
// arithmetic: a value is an unevaluated sum hi + lo of two float64, kept exact
// by the error-free sum of Knuth and Moller and the error-free product of a
// fused multiply-add (Dekker's algorithms; Hida, Li and Bailey's double-double
// library describes the same operations). The constants come from series:
// ln 2 = 2 atanh(1/3), pi from Machin's formula, ln(base) by Newton's
// iteration on exp, and exp by its Taylor series after reducing the argument
// by multiples of ln 2 and ten halvings.
#include <cmath>
#include <cstdint>

#include "sr_kernels.h"

namespace {

struct DD {
  double hi, lo;
};

DD two_sum(double a, double b) {   // a + b = s + e exactly
  const double s = a + b;
  const double bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}

DD fast_two_sum(double a, double b) {   // |a| >= |b|
  const double s = a + b;
  return {s, b - (s - a)};
}

DD two_prod(double a, double b) {   // a * b = p + e exactly
  const double p = a * b;
  return {p, std::fma(a, b, -p)};
}

DD dd(double x) { return {x, 0.0}; }
DD neg(DD a) { return {-a.hi, -a.lo}; }
DD ldexp_dd(DD a, int e) { return {std::ldexp(a.hi, e), std::ldexp(a.lo, e)}; }

DD add(DD a, DD b) {
  DD s = two_sum(a.hi, b.hi);
  const DD t = two_sum(a.lo, b.lo);
  s.lo += t.hi;
  s = fast_two_sum(s.hi, s.lo);
  s.lo += t.lo;
  return fast_two_sum(s.hi, s.lo);
}

DD mul(DD a, DD b) {
  DD p = two_prod(a.hi, b.hi);
  p.lo += a.hi * b.lo + a.lo * b.hi;
  return fast_two_sum(p.hi, p.lo);
}

DD div(DD a, DD b) {   // long division: three float64 quotient digits
  const double q1 = a.hi / b.hi;
  DD r = add(a, neg(mul(b, dd(q1))));
  const double q2 = r.hi / b.hi;
  r = add(r, neg(mul(b, dd(q2))));
  const double q3 = r.hi / b.hi;
  return add(fast_two_sum(q1, q2), dd(q3));
}

// sum_{k>=0} (-1)^k / ((2k+1) x^(2k+1)) = atan(1/x) (alternate = true) or
// atanh(1/x) (alternate = false), for an integer x >= 3.
DD arc_series(int x, bool alternate) {
  const DD inv = div(dd(1.0), dd(x));
  const DD inv2 = mul(inv, inv);
  DD power = inv, sum = dd(0.0);
  for (int k = 0; k < 200; ++k) {
    const DD term = div(power, dd(2.0 * k + 1.0));
    sum = add(sum, (alternate && (k & 1)) ? neg(term) : term);
    if (std::fabs(term.hi) < 1e-40) break;
    power = mul(power, inv2);
  }
  return sum;
}

DD ln2_dd() { return ldexp_dd(arc_series(3, false), 1); }   // 2 atanh(1/3)

DD pi_dd() {   // Machin: pi = 16 atan(1/5) - 4 atan(1/239)
  return add(ldexp_dd(arc_series(5, true), 4), neg(ldexp_dd(arc_series(239, true), 2)));
}

DD exp_dd(DD x, DD ln2) {
  const double k = std::nearbyint(x.hi / ln2.hi);
  DD r = add(x, neg(mul(ln2, dd(k))));   // |r| <= ln2 / 2
  r = ldexp_dd(r, -10);
  // s = e^r - 1 by its Taylor series
  DD term = r, s = r;
  for (int n = 2; n < 40; ++n) {
    term = div(mul(term, r), dd(n));
    s = add(s, term);
    if (std::fabs(term.hi) <= 1e-36 * std::fabs(s.hi)) break;
  }
  // e^(2y) - 1 = 2 (e^y - 1) + (e^y - 1)^2, ten times
  for (int i = 0; i < 10; ++i) s = add(ldexp_dd(s, 1), mul(s, s));
  return ldexp_dd(add(dd(1.0), s), static_cast<int>(k));
}

DD log_dd(double x, DD ln2) {   // Newton on exp: y <- y + x e^(-y) - 1
  DD y = dd(std::log(x));
  for (int it = 0; it < 3; ++it) y = add(y, add(mul(dd(x), exp_dd(neg(y), ln2)), dd(-1.0)));
  return y;
}

// round(c * 2^96) for 0 <= c < 1, as the high 64 and low 32 bits.
void to_fixed96(DD c, uint64_t* U, uint32_t* E) {
  const double h = std::ldexp(c.hi, 96);   // below 2^96
  const double hr = std::nearbyint(h);     // h itself once h >= 2^52
  const double top = std::floor(std::ldexp(hr, -64));
  const double low = hr - std::ldexp(top, 64);   // exact: the bits of hr below 2^64
  unsigned __int128 v = (static_cast<unsigned __int128>(static_cast<uint64_t>(top)) << 64) +
                        static_cast<unsigned __int128>(static_cast<uint64_t>(low));
  // what hr dropped plus the low part: at most about 2^43 in magnitude
  const long long l = std::llround(std::ldexp(c.lo, 96) + (h - hr));
  v = l >= 0 ? v + static_cast<unsigned __int128>(l) : v - static_cast<unsigned __int128>(-l);
  *U = static_cast<uint64_t>(v >> 32);
  *E = static_cast<uint32_t>(v);
}

}  // namespace

namespace sr {

void rope_phase_table(float base, int head_dim, RopePhase* out) {
  const DD ln2 = ln2_dd();
  const DD two_pi = ldexp_dd(pi_dd(), 1);
  const DD ln_base = log_dd(static_cast<double>(base), ln2);
  const int dh = 2 * (head_dim / 6);
  const int dims[3] = {head_dim - 2 * dh, dh, dh};
  int p = 0;
  for (int a = 0; a < 3; ++a) {
    for (int i = 0; i < dims[a] / 2; ++i, ++p) {
      // omega = exp(-(2i/d_axis) ln base); c = omega / (2 pi) turns per step
      const DD expo = div(dd(-2.0 * i), dd(dims[a]));
      const DD omega = exp_dd(mul(expo, ln_base), ln2);
      to_fixed96(div(omega, two_pi), &out->turn_hi[p], &out->turn_lo[p]);
      out->axis[p] = static_cast<int8_t>(a);
    }
  }
  for (; p < kMaxPairs; ++p) {
    out->turn_hi[p] = 0;
    out->turn_lo[p] = 0;
    out->axis[p] = 0;
  }
  // 2 pi / 2^32 as two floats: the radians of one unit of a phase's high word
  const DD rad = ldexp_dd(two_pi, -32);
  out->rad_hi = static_cast<float>(rad.hi);
  out->rad_lo = static_cast<float>(add(rad, dd(-static_cast<double>(out->rad_hi))).hi);
}

}  // namespace sr
