// Device helpers shared by the frame-loop kernels: bounded waits that honour
// a grid-wide abort flag, counter atomics with explicit memory order, f16
// packing, and the per-warp RMSNorm + RoPE and score reduction of attention.
// A params type passed to the waits has int* members abort_flag and status
// and a long long spin_limit (clock64 ticks).
#pragma once

#include "qp_common.cuh"
#include "qp_internal.h"
#include "qp_ptx.cuh"

namespace qp {
namespace {

// ------------------------------------------------------------------ waits
template <class Par>
__device__ __forceinline__ void abort_all(const Par& p) {
  set_status(p.status, QP_ERR_TIMEOUT);
  atomicExch(p.abort_flag, 1);
}
template <class Par>
__device__ __forceinline__ bool aborted(const Par& p) { return *(volatile int*)p.abort_flag != 0; }

// Until *ctr >= want (acquire), bounded.  After two misses each poll is
// spaced by a short sleep, which eases the load the waiting threads of every
// CTA put on the counters' L2 lines (about 1 % per step, measured).
template <class Par>
__device__ bool poll_geq(const Par& p, const unsigned* ctr, unsigned want) {
  if (ld_acquire_u32(ctr) >= want) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (ld_acquire_u32(ctr) >= want) return true;
    if (it > 2) __nanosleep(32);
    if ((it & 63) == 0) {
      if (aborted(p)) return false;
      if (clock64() - t0 > p.spin_limit) { abort_all(p); return false; }
    }
  }
}

// mbarrier phase wait, bounded, abandoning when the grid aborts.
template <class Par>
__device__ bool mwait(const Par& p, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (aborted(p)) return false;
      if (clock64() - t0 > p.spin_limit) { abort_all(p); return false; }
    }
  }
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A relaxed add: after fence_acq_rel_gpu(), a run of these releases the
// writes before the fence as each red.release would, with one fence.
__device__ __forceinline__ void red_relaxed_add(unsigned* p, unsigned v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Fetch-and-add with acquire-release semantics at GPU scope: publishes this
// CTA's earlier writes (ordered before it by bar.sync) and, for the caller
// that completes a count, makes every earlier contributor's writes visible.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// ------------------------------------------------------ f16 operand range
// A GEMM operand row built from the residual stream (or from H) is
// multiplied by 2^-e before its f16 conversion, and the GEMM's f32 result
// by 2^e after it (both exact), so that rows of any magnitude stay inside
// f16's range (65504).  e comes from the mean square ms of a reference row
// known before the operand is built -- the row itself where it is complete,
// else the same frame's most recent complete residual row: 2^-e brings that
// row's RMS into [2^-5, 2^-4), or e = 0 (no scaling) when the RMS is below
// 2^-5.  A row may grow far past its reference within one sublayer before
// 2^-e * |x| * |w_norm| reaches 65504, and f16's relative precision does not
// depend on the scale above its smallest normal value (2^-14).
__device__ __forceinline__ int range_exp(float ms) {
  const int E = int((__float_as_uint(ms) >> 23) & 255u) - 127;   // floor(log2(ms)) for ms >= 2^-126
  const int e = (E >> 1) + 5;                                      // floor(log2(RMS)) + 5
  return e < 0 ? 0 : (e > 100 ? 100 : e);
}
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(uint32_t(127 + e) << 23); }   // |e| <= 126

__device__ __forceinline__ uint2 pack4_f16(float a, float b, float c, float d) {
  return make_uint2(uint32_t(f32_to_f16_bits(a)) | (uint32_t(f32_to_f16_bits(b)) << 16),
                    uint32_t(f32_to_f16_bits(c)) | (uint32_t(f32_to_f16_bits(d)) << 16));
}
__device__ __forceinline__ float4 unpack4_f16(uint2 v) {
  return make_float4(f16_bits_to_f32(v.x & 0xffff), f16_bits_to_f32(v.x >> 16), f16_bits_to_f32(v.y & 0xffff),
                     f16_bits_to_f32(v.y >> 16));
}


// RMSNorm of a 128-vector held as 4 values per lane, then rotate-half RoPE
// at position pos (pairs (i, i+64) sit in lanes l and l^16).
__device__ __forceinline__ float4 norm_rope(float4 x, const float* nw, float eps, const float2* cs, int lane) {
  const float ss = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
  const float r = rsqrtf(ss / 128.f + eps);
  const float4 w = *reinterpret_cast<const float4*>(nw + lane * 4);
  float v[4] = {x.x * r * w.x, x.y * r * w.y, x.z * r * w.z, x.w * r * w.w};
  float o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float partner = __shfl_xor_sync(0xffffffffu, v[e], 16);
    const float2 c = cs[(lane * 4 + e) & 63];
    o[e] = lane < 16 ? v[e] * c.x - partner * c.y : v[e] * c.x + partner * c.y;
  }
  return make_float4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// ------------------------------------------------------ top-k selection
// The top_k-th largest of the order keys keys[0..V) in shared memory, by a
// most-significant-digit radix select over four 8-bit digits (all NT
// consumer threads of the CTA, which meet at named barrier `bar`; hist has
// 256 entries, sel 2).  Returns that key; `remaining` says how many keys
// equal to it belong to the top_k (the first ones in index order).  Each
// digit is chosen by one warp: lane l holds the 8 bins 255-8l .. 248-8l, a
// shuffle prefix sum gives every lane the count above its bins, and the lane
// whose range reaches `remaining` picks the digit.
template <int NT>
__device__ uint32_t topk_kth_key(const uint32_t* keys, int V, int top_k, int* hist, int* sel, int bar,
                                 int& remaining) {
  const int t = threadIdx.x, lane = t & 31;
  uint32_t prefix = 0, mask = 0;
  remaining = top_k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = t; i < 256; i += NT) hist[i] = 0;
    named_bar(bar, NT);
    for (int i = t; i < V; i += NT) {
      const uint32_t kk = keys[i];
      if ((kk & mask) == prefix) atomicAdd(&hist[(kk >> shift) & 255], 1);
    }
    named_bar(bar, NT);
    if (t < 32) {
      int c[8], s = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { c[i] = hist[255 - 8 * lane - i]; s += c[i]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = incl - s;
      if (excl < remaining && remaining <= incl) {   // exactly one lane
        int cum = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + c[i] >= remaining) { sel[0] = 255 - 8 * lane - i; sel[1] = remaining - cum; break; }
          cum += c[i];
        }
      }
      if (lane == 31 && incl < remaining) { sel[0] = 0; sel[1] = remaining - incl; }   // not reached for top_k <= V
    }
    named_bar(bar, NT);
    prefix |= uint32_t(sel[0]) << shift;
    mask |= 255u << shift;
    remaining = sel[1];
    named_bar(bar, NT);   // sel and hist are rewritten by the next digit
  }
  return prefix;
}

// Exclusive prefix sum of v over the NT threads in thread order (CTA-wide;
// wtot holds NT / 32 ints).  Ends with the barrier that publishes the warp
// totals; the caller's next barrier must come before wtot is rewritten.
template <int NT>
__device__ int block_exclusive_scan(int v, int* wtot, int bar) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wtot[warp] = incl;
  named_bar(bar, NT);
  int off = 0;
  for (int w = 0; w < warp; ++w) off += wtot[w];
  return off + incl - v;
}

// Sixteen warp-wide sums: lane l ends with the total over all 32 lanes of
// v[(l >> 1) & 15] (lanes 2i and 2i + 1 both hold sum i).  Four halving
// exchanges, then the lane pairs meet.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 16; o >= 2; o >>= 1) {
    const int c = o >> 1;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c; ++i) {
      const float send = upper ? v[i] : v[i + c];
      const float keep = upper ? v[i + c] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

}  // namespace
}  // namespace qp
