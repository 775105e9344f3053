// common.cuh -- device helpers shared by the kernels: scale-factor addressing, E8M0 / E4M3
// scale logic in integer arithmetic, device error reporting and bounded waits.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace bsg {

constexpr uint32_t kErrTimeout = 0x1u;     // matches BSG_DEVERR_TIMEOUT
constexpr uint32_t kErrBadOffsets = 0x2u;  // matches BSG_DEVERR_BAD_OFFSETS
constexpr uint32_t kErrBadPointers = 0x4u;  // matches BSG_DEVERR_BAD_POINTERS

// A pipeline wait longer than this is taken as a hang: the kernel records an error and
// leaves instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Byte offset of (row r, scale block kb, batch l) in the 128x4 scale-factor atom layout
// (physical (batch, MT, KT, 32, 4, 4) bytes, row r = 128*mt + 32*i1 + i0, block kb = 4*kt + k0).
__device__ __forceinline__ uint64_t sf_offset(uint64_t r, uint64_t kb, uint64_t l, uint64_t mt_n, uint64_t kt_n) {
  return ((((l * mt_n + (r >> 7)) * kt_n + (kb >> 2)) * 32 + (r & 31)) * 4 + ((r & 127) >> 5)) * 4 + (kb & 3);
}

// E8M0 code of the smallest power of two 2^e with v <= 448 * 2^e, clamped to [0, 254].
// v = 1.f * 2^E (normal fp32): 448 * 2^e = 1.75 * 2^(e+8), so e = E - 8 when 1.f <= 1.75
// (mantissa field <= 0x600000) and E - 7 otherwise.  Zero and subnormal v give code 0
// (their e is below -127).
__device__ __forceinline__ uint32_t e8m0_ceil_code(float v) {
  const uint32_t bits = __float_as_uint(v);
  const int exp_field = static_cast<int>((bits >> 23) & 0xFF);
  if (!(v > 0.0f) || exp_field == 0) return 0;
  const uint32_t mant = bits & 0x7FFFFFu;
  const int e = (exp_field - 127) - (mant <= 0x600000u ? 8 : 7);
  const int code = e + 127;
  return static_cast<uint32_t>(code < 0 ? 0 : (code > 254 ? 254 : code));
}

// 2^(127 - code) as fp32 (the reciprocal of an E8M0 scale), code in [0, 254].
__device__ __forceinline__ float e8m0_inv_scale(uint32_t code) {
  return code <= 253 ? __uint_as_float((254u - code) << 23) : __uint_as_float(0x00400000u);
}

// Value of an E4M3 code with the sign bit ignored (an unsigned scale), code 0..0x7E.
__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xF, m = code & 7;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));    // (1 + m/8) * 2^(e-7)
}

// Device error record in the first bytes of a call's workspace (32-bit words):
//   words 0-1  the error bits (word 0) tagged with the epoch of the call that set them (word 1),
//              updated together by one 64-bit atomic;
//   word 2     the epoch of the last call whose kernel ran (every CTA stores it at its start).
// Every call gets a fresh nonzero epoch from the library, and the host takes the bits as the
// last call's only when words 1 and 2 agree, so no call has to clear the workspace before its
// kernel runs.
struct ErrSink {
  uint32_t* ws;    // the workspace (8-byte aligned), or nullptr
  uint32_t epoch;  // this call's epoch
};

// Marks the workspace as used by this call (any thread of every CTA may do it; same value).
__device__ __forceinline__ void mark_call(const ErrSink& e) {
  if (e.ws != nullptr) *reinterpret_cast<volatile uint32_t*>(e.ws + 2) = e.epoch;
}

// ORs `bits` into this call's error bits (replacing bits a previous call left behind).
__device__ __forceinline__ void report_error(const ErrSink& e, uint32_t bits) {
  if (e.ws == nullptr) return;
  unsigned long long* w = reinterpret_cast<unsigned long long*>(e.ws);
  const unsigned long long tag = static_cast<unsigned long long>(e.epoch) << 32;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w), assumed;
  do {
    assumed = old;
    const unsigned long long nv = ((assumed >> 32) == e.epoch) ? (assumed | bits) : (tag | bits);
    old = atomicCAS(w, assumed, nv);
  } while (old != assumed);
}

// Waits for phase `parity` of `bar` to complete.  Gives up (returns false) when another
// role of the CTA has aborted or after kWaitLimitNs, in which case it records a timeout
// and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             const ErrSink& err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        report_error(err, kErrTimeout);
        return false;
      }
    }
  }
}

// Same wait without the abort flag (used while tearing down after an abort).
__device__ __forceinline__ bool wait_bounded_plain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

}  // namespace bsg
