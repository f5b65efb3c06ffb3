// Internal definitions shared by the library's translation units: the layout
// of the derived tree tables, device status helpers and small numeric helpers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "tv.h"

namespace tv {

// Programmatic dependent launch: let the next kernel on the stream start its
// own set-up, and wait until the previous kernel has finished and its writes
// are visible.  Both are no-ops for a kernel launched without the attribute.
// A kernel that never calls pdl_trigger lets the next one start as its
// blocks exit.  The attention split kernel and GDN verify trigger early: both
// run at most one CTA per SM, so an early successor only takes SMs they do
// not use (measured: 1.8 % per round from GDN).  The attention tail triggers
// right after its wait: its CTAs leave SMs free, where the next kernel can
// start (0.2-0.3 % per round).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// A bounded wait gives up after this many SM clocks (about a second).
constexpr long long kWaitCycles = 1LL << 31;

// ----------------------------------------------------------------------------
// derived tree tables (written by tv_tree_prepare, read by the other calls)
// ----------------------------------------------------------------------------
struct SeqInfo {
  int32_t n;          // nodes of this sequence's tree (0 = invalid tree)
  int32_t off;        // first global node index
  int32_t max_depth;  // deepest node
  int32_t max_slot;   // saved-state slots the recurrent traversal needs
  int32_t n_seg;      // segments of the recurrent traversal (seg entries)
  int32_t pad[3];
};

struct MetaView {
  SeqInfo* seq;     // [TV_MAX_SEQ]
  uint64_t* anc;    // [n_total] ancestor-or-self bitmask (sequence-local bits)
  int32_t* depth;   // [n_total]
  int32_t* sched;   // [n_total] recurrent traversal, per sequence at off..off+n-1
  int32_t* seg;     // [n_total] segments of the traversal, per sequence at off..off+n_seg-1
  int8_t* anc_at;   // [n_total][TV_MAX_PATH] local index of the ancestor at each depth
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

__host__ __device__ inline size_t meta_bytes(int n_total) {
  const size_t n = static_cast<size_t>(n_total);
  return align16(sizeof(SeqInfo) * TV_MAX_SEQ) + align16(8 * n) + 3 * align16(4 * n) +
         align16(TV_MAX_PATH * n);
}

__host__ __device__ inline MetaView meta_view(void* base, int n_total) {
  const size_t n = static_cast<size_t>(n_total);
  char* p = static_cast<char*>(base);
  MetaView m;
  m.seq = reinterpret_cast<SeqInfo*>(p);
  p += align16(sizeof(SeqInfo) * TV_MAX_SEQ);
  m.anc = reinterpret_cast<uint64_t*>(p);
  p += align16(8 * n);
  m.depth = reinterpret_cast<int32_t*>(p);
  p += align16(4 * n);
  m.sched = reinterpret_cast<int32_t*>(p);
  p += align16(4 * n);
  m.seg = reinterpret_cast<int32_t*>(p);
  p += align16(4 * n);
  m.anc_at = reinterpret_cast<int8_t*>(p);
  return m;
}

// Recurrent traversal.  A visit: [0,8) local node, bit 24 = node has
// children.  A segment of consecutive visits: [0,8) first visit, [8,16)
// visits, [16,24) source of the state the segment starts from (0 = the state
// already in registers, 1+k = saved slot k), [24,32) slot the state is saved
// to after the segment's last visit (0 = none, 1+k = slot k).
constexpr int kMaxSlots = 5;  // a tree of <= 64 nodes never needs more (see tree.cu)
__host__ __device__ inline int32_t visit_encode(int node, int has_children) { return node | (has_children << 24); }
__host__ __device__ inline int32_t seg_encode(int first, int count, int src, int save) {
  return first | (count << 8) | (src << 16) | (save << 24);
}

// ----------------------------------------------------------------------------
// device status word: the first error code wins; later calls become no-ops
// ----------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}
__device__ __forceinline__ bool status_bad(const int32_t* st) {
  return st != nullptr && *reinterpret_cast<const volatile int32_t*>(st) != 0;
}

// ----------------------------------------------------------------------------
// element conversion
// ----------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Output gate of the attention front end: x * sigmoid(g), with the sigmoid
// as 1 / (1 + e^-g) (CUDA's expf, IEEE add and divide); the same function for
// verify and decode rows.
__device__ __forceinline__ float gate_mul(float x, float g) {
  return __fmul_rn(x, __fdiv_rn(1.f, __fadd_rn(1.f, expf(-g))));
}

// Plain stores to global memory, as explicit global-space instructions.
__device__ __forceinline__ void store_global(float* p, float v) { asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(v)); }
__device__ __forceinline__ void store_global(__nv_bfloat16* p, __nv_bfloat16 v) {
  asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(__bfloat16_as_ushort(v)));
}

// bf16 halves of a packed word, exactly
// Packed fp32 pairs: each lane of an f32x2 operation rounds as its scalar
// counterpart does.
typedef unsigned long long f2_t;  // two fp32 values in one 64-bit register

__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_dup(float x) {
  f2_t d;
  asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(x));
  return d;
}
__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_unpack(f2_t a, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
}
__device__ __forceinline__ float f2_hsum(f2_t a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return __fadd_rn(lo, hi);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace tv
