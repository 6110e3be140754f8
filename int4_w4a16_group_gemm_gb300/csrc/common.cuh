// Device-side helpers shared by the W4A16 kernels: status word, bounded
// mbarrier waits, bulk (TMA) copies and small conversions. sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w4a16.h"

namespace w4a16 {

// ---------------------------------------------------------------- status
// Kernels record the first error they see in a per-device status word whose
// address the host passes in (no relocatable device code needed).
__device__ __forceinline__ void record_status(int *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Bounds checks of the W4A16_DEBUG build: W4A16_IN_BOUNDS(cond, status)
// is true when the access it guards stays inside its buffer; otherwise it
// records W4A16_ERR_BOUNDS in the status word and is false, so the caller
// skips the access. In the release build it is `true` and compiles away.
#ifdef W4A16_DEBUG
__device__ __forceinline__ bool w4a16_in_bounds(bool ok, int *status) {
  if (!ok) record_status(status, W4A16_ERR_BOUNDS);
  return ok;
}
#define W4A16_IN_BOUNDS(cond, status) (::w4a16::w4a16_in_bounds((cond), (status)))
#else
#define W4A16_IN_BOUNDS(cond, status) true
#endif

// Wall-clock bound for every spin-wait, in nanoseconds (~1 s).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` (mbarrier.try_wait may suspend the
// thread for a while when the phase is not complete; test_wait never does).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps (issuing nothing)
// until the phase completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after
// kWaitLimitNs. Returns false on timeout (the caller records it). The wait
// spins: a suspend-time hint or a sleep between checks measurably delays
// the wake-up on this GPU, and the pipelines here are latency-bound.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// As mbar_wait, for a waiter with slack: polls without suspending and
// sleeps about `sleep_ns` between polls, so that while it waits it takes
// (almost) no issue slots from the warps on its scheduler. Meant for one
// lane per warp.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t *bar, uint32_t parity,
                                                  uint32_t sleep_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(sleep_ns);
    if (mbar_test_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// As mbar_wait, but also gives up (returning false) once `*abort` becomes
// nonzero: another warp of the CTA has already timed out, so the phase may
// never complete. The flag is polled between batches of try_waits.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity,
                                                   const volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort != 0 || globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- bulk copy
// 1-D bulk copy global -> shared, completion signalled on `bar` as tx bytes.
// dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch. launch_dependents lets the next kernel on
// the stream start launching; wait blocks until the previous kernel has
// completed and its memory is visible. Both are no-ops for a kernel
// launched without the programmatic-serialisation attribute.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// SiLU in fp32: g * sigmoid(g).
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Store element i of the output: fp32, or rounded to bf16 (to nearest,
// ties to even) when `bf16` is set and y holds 16-bit elements.
__device__ __forceinline__ void store_y(void *y, size_t i, float v, int bf16) {
  if (bf16)
    static_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float *>(y)[i] = v;
}

// ---------------------------------------------------------------- numbers
// `v`, returned through a warp shuffle so that the compiler can neither
// fold it into an instruction immediate nor re-create it with a move before
// every use (both cost instructions on the unpack's critical pipes). All 32
// lanes of the warp must call it together.
__device__ __forceinline__ uint32_t opaque_u32(uint32_t v) {
  return __shfl_sync(0xFFFFFFFFu, v, 0);
}
__device__ __forceinline__ float opaque_f32(float v) { return __shfl_sync(0xFFFFFFFFu, v, 0); }

// Nibble unpack to fp32 without integer->float conversions. A packed word
// holds nibbles n0..n7 (nibble j in bits 4j..4j+3). For c in 0..3 the
// nibbles c and c+4 are moved into the two fp16 halves of one register:
//   h = (src & mask_c) | 0x64006400,  src = word (c < 2) or word >> 8 (c >= 2),
//   mask_c = 0x000F000F (c even) or 0x00F000F0 (c odd),
// so each half is the fp16 number 1024 + n (c even) or 1024 + 16 n (c odd),
// exact. One mixed-precision add per half, f32(half) + bias with bias =
// -1032 (c even) or -1152 (c odd), then gives (n - 8) or 16 (n - 8) as an
// exact fp32 number; the activations of odd classes are pre-multiplied by
// 1/16 (an exact scaling). The constants live in registers (NibbleConsts):
// as immediates the compiler would spend extra instructions on them.
struct NibbleConsts {
  uint32_t magic;  // 0x64006400: two fp16 1024.0
  float bias_even, bias_odd;
};
__device__ __forceinline__ NibbleConsts make_nibble_consts() {
  return {opaque_u32(0x64006400u), opaque_f32(-1032.0f), opaque_f32(-1152.0f)};
}
// Both nibbles of class c of `word` as exact fp32 values (n - 8) * (c odd ?
// 16 : 1), in the low and high halves of a packed fp32 pair.
template <int C>
__device__ __forceinline__ uint64_t nibble_pair(uint32_t word, uint32_t word_sh8,
                                                const NibbleConsts &k) {
  const uint32_t src = C < 2 ? word : word_sh8;
  const uint32_t h = (src & ((C & 1) ? 0x00F000F0u : 0x000F000Fu)) | k.magic;
  const float bias = (C & 1) ? k.bias_odd : k.bias_even;
  uint64_t r;
  asm("{\n\t.reg .f16 lo, hi;\n\t.reg .f32 a, b;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 a, lo, %2;\n\tadd.rn.f32.f16 b, hi, %2;\n\tmov.b64 %0, {a, b};\n\t}"
      : "=l"(r)
      : "r"(h), "f"(bias));
  return r;
}
// Pre-scale factor of the activation matching a class-c nibble.
__host__ __device__ constexpr float nibble_prescale(int c) { return (c & 1) ? 0.0625f : 1.0f; }

// ---------------------------------------------------------------- fp32 pairs
// Packed fp32 pairs: Blackwell's add/fma.f32x2 do two independent fp32
// operations (each rounded exactly like the scalar one) per instruction.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ---------------------------------------------------------------- unpack
// Exact fp32 (nibble - 8) of the same nibble position of two packed words,
// as the two halves of one packed fp32 pair, with one logic instruction per
// value and one packed subtract per pair:
//   nibble j of a word sits in bits 4j..4j+3. For j <= 4 those bits lie in
//   the fp32 mantissa; ORing them into the bits of 2^(23-4j) (mantissa 0)
//   gives the fp32 number 2^(23-4j) + nibble exactly (the mantissa's unit
//   in the last place is 2^(-4j) there, times 2^(4j) for the nibble's
//   position). Subtracting 2^(23-4j) + 8 leaves nibble - 8, exact.
//   Nibbles 5..7 are taken from the word shifted right by 12, where they sit
//   at positions 2..4.
// The GPU's logic pipe runs at half the rate of its fp32 pipe, so the
// unpack is written as explicit lop3 ((w & mask) | magic in one
// instruction; the compiler otherwise emits an AND and an OR) and packed
// fp32 arithmetic; values never pass through fp16 halves, whose extraction
// costs further logic instructions.
struct PairUnpack {
  uint32_t magic[5];  // fp32 bits of 2^(23-4j)
};

__device__ __forceinline__ PairUnpack make_pair_unpack() {
  PairUnpack k;
#pragma unroll
  for (int j = 0; j < 5; ++j) k.magic[j] = opaque_u32(static_cast<uint32_t>(127 + 23 - 4 * j) << 23);
  return k;
}

// The packed bias -(2^(23-4j) + 8) of nibble position j (a compile-time
// constant, which the compiler may keep outside the register file).
template <int J>
__device__ __forceinline__ uint64_t pair_bias() {
  constexpr float b = -static_cast<float>((1u << (23 - 4 * J)) + 8u);
  return (static_cast<uint64_t>(__float_as_uint(b)) << 32) | __float_as_uint(b);
}

template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t o) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(o));
  return d;
}

__device__ __forceinline__ uint64_t pair_u32(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

// v[j] = (nibble j of a - 8, nibble j of b - 8), j = 0..7.
__device__ __forceinline__ void unpack8_pair(uint32_t a, uint32_t b, const PairUnpack &k,
                                             uint64_t (&v)[8]) {
  const uint32_t a12 = a >> 12, b12 = b >> 12;
  v[0] = add_f32x2(pair_u32(lop_and_or<0xFu>(a, k.magic[0]), lop_and_or<0xFu>(b, k.magic[0])), pair_bias<0>());
  v[1] = add_f32x2(pair_u32(lop_and_or<0xF0u>(a, k.magic[1]), lop_and_or<0xF0u>(b, k.magic[1])), pair_bias<1>());
  v[2] = add_f32x2(pair_u32(lop_and_or<0xF00u>(a, k.magic[2]), lop_and_or<0xF00u>(b, k.magic[2])), pair_bias<2>());
  v[3] = add_f32x2(pair_u32(lop_and_or<0xF000u>(a, k.magic[3]), lop_and_or<0xF000u>(b, k.magic[3])), pair_bias<3>());
  v[4] = add_f32x2(pair_u32(lop_and_or<0xF0000u>(a, k.magic[4]), lop_and_or<0xF0000u>(b, k.magic[4])), pair_bias<4>());
  v[5] = add_f32x2(pair_u32(lop_and_or<0xF00u>(a12, k.magic[2]), lop_and_or<0xF00u>(b12, k.magic[2])), pair_bias<2>());
  v[6] = add_f32x2(pair_u32(lop_and_or<0xF000u>(a12, k.magic[3]), lop_and_or<0xF000u>(b12, k.magic[3])), pair_bias<3>());
  v[7] = add_f32x2(pair_u32(lop_and_or<0xF0000u>(a12, k.magic[4]), lop_and_or<0xF0000u>(b12, k.magic[4])), pair_bias<4>());
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

}  // namespace w4a16
