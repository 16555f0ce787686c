// Inline-PTX building blocks for the sm_103a tensor-core kernels: mbarriers,
// TMA tensor loads, tcgen05 TMEM allocation / MMA / commit / load / store and
// the shared-memory matrix and instruction descriptors, written from the
// public PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace jfa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Gives up after `limit` clock cycles or as soon as another
// role of the CTA has given up (*abort != 0); on giving up it raises *abort
// and records JFA_ERR_TIMEOUT in the device status word.  Returns false if
// the wait did not complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const long long limit = 4000000000LL;  // ~2 s at 2 GHz
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > limit) {
        *abort = 1;
        atomicExch(status, (int)JFA_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait used when a role leaves its loop, normally or after giving up: it
// ignores the abort flag, so that a role that gave up still waits for its own
// asynchronous operations (MMAs, TMA loads) to land before the CTA frees TMEM and
// exits.  They always complete, so the limit is only a guard.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const long long limit = 4000000000LL;  // ~2 s at 2 GHz
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && clock64() - t0 > limit) {
      atomicExch(status, (int)JFA_ERR_TIMEOUT);
      return false;
    }
  }
}

// A producer's loads into a ring of `stages` stages with `loads` loads issued in
// stage order: waits until the last load into every stage has landed.
__device__ __forceinline__ void drain_ring(uint32_t full_bar0, uint32_t stages, uint32_t loads,
                                           int* status) {
  for (uint32_t s = 0; s < stages && s < loads; ++s) {
    const uint32_t count = (loads - s + stages - 1) / stages;  // loads into stage s
    mbar_wait_drain(full_bar0 + 8u * s, (count - 1) & 1u, status);
  }
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// ---------------------------------------------------------------- TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// MMA issue.  The issuing warp runs converged: all 32 lanes compute the same
// descriptors (so they stay warp-uniform) and execute these helpers together; one
// lane, chosen by elect.sync, issues the instruction.  Issuing from inside an
// `if (lane == 0)` branch instead costs the issuing thread markedly more per MMA.
// elect.sync picks the lowest active lane, the same lane every time, so a commit
// covers the MMAs issued before it.

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate), one CTA.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x K, bf16) read from tensor memory, one row per
// lane, two consecutive K elements packed per 32-bit column (K = 16 -> 8 columns).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by the issuing lane has
// completed (warp-collective, like the MMA helpers).
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
      : "memory");
}
// An MMA issuer's drain when it leaves its loop: a commit of everything it issued
// to a barrier of its own (count 1, used once), and a wait for it (warp-collective).
__device__ __forceinline__ void mma_drain(uint32_t drain_bar, int* status) {
  mma_commit(drain_bar);
  mbar_wait_drain(drain_bar, 0, status);
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
// The tile is a stack of 1024-byte swizzle atoms of 8 rows x 128 bytes, as
// written by a TMA load with CU_TENSOR_MAP_SWIZZLE_128B into 1024-aligned smem.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo_bytes,
                                               uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, M x N tile.
// a_mn / b_mn: operand stored MN-major (1) instead of K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                    // D format: f32
         | (1u << 7)                  // A format: bf16
         | (1u << 10)                 // B format: bf16
         | ((uint32_t)a_mn << 15)     // A major-ness
         | ((uint32_t)b_mn << 16)     // B major-ness
         | ((uint32_t)(N >> 3) << 17) // N / 8
         | ((uint32_t)(M >> 4) << 24);// M / 16
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed two-wide fp32 arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n.reg .b64 ra, rb, rc, rd;\n"
      "mov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\nmov.b64 rc, {%6, %7};\n"
      "fma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 r;
  asm("{\n.reg .b64 ra, rb, rd;\n"
      "mov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "mul.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 r;
  asm("{\n.reg .b64 ra, rb, rd;\n"
      "mov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "add.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float tanh_approx(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
  return t;
}

// sigmoid(u) = 1/2 + tanh(u/2)/2: one MUFU operation (tanh.approx) instead of
// an exp2 and a reciprocal.  Exact 0 for the masked (hugely negative) scores.
__device__ __forceinline__ float sigmoid_fast(float u) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * u));
  return fmaf(0.5f, t, 0.5f);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Elementwise product of two packed bf16 pairs, rounded once to bf16 (a fused multiply-add
// with -0 as the addend, so a product of +0 stays +0).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(0x80008000u));
  return r;
}
// 32-byte global store (dst must be 32-byte aligned)
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* r) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// 32 floats times f as bf16 to dst: 32-byte stores when dst is 32-byte aligned
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float* x, float f) {
  uint32_t w[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) w[t] = pack_bf16(x[2 * t] * f, x[2 * t + 1] * f);
  if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
    st_global_v8(dst, w);
    st_global_v8(dst + 16, w + 8);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int t = 0; t < 4; ++t) d[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
  }
}
// 16 floats times f as bf16 to dst (32 bytes): one 32-byte store when dst is 32-byte aligned
__device__ __forceinline__ void store16_bf16(__nv_bfloat16* dst, const float* x, float f) {
  uint32_t w[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) w[t] = pack_bf16(x[2 * t] * f, x[2 * t + 1] * f);
  if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
    st_global_v8(dst, w);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}
// n (16 or a multiple of 32) floats times f as bf16 to dst
template <int N>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* dst, const float* x, float f) {
  static_assert(N == 16 || N % 32 == 0, "16 or whole 32-column chunks");
  if constexpr (N == 16) {
    store16_bf16(dst, x, f);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) store32_bf16(dst + 32 * c, x + 32 * c, f);
  }
}
// n (16 or a multiple of 32) consecutive fp32 columns of this thread's TMEM lane
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
  static_assert(N == 16 || N % 32 == 0, "16 or whole 32-column chunks");
  if constexpr (N == 16) {
    tmem_ld16(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_ld32(taddr + 32 * c, v + 32 * c);
  }
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------- rotary embedding
// The pair (x0, x1) of a bf16x2 word turned by the angle with cosine c and sine s:
// (x0 c - x1 s, x0 s + x1 c), rounded to bf16.
__device__ __forceinline__ uint32_t rope_rotate_word(uint32_t w, float c, float s) {
  const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
  return pack_bf16(fmaf(x0, c, -x1 * s), fmaf(x0, s, x1 * c));
}

// The rotary position embedding of a tile in shared memory, in place: row r at position
// pos0 + r, its columns (2i, 2i+1) turned by the angle whose (cos, sin) is
// table[(pos0 + r) * (D/2) + i].  The tile is D/64 boxes of 64 bf16 columns, 16 KB apart,
// each a stack of 128-byte-swizzled 8-row atoms (as a TMA load with 128-byte swizzle
// writes them).  Each lane fences its writes to the async proxy, so that once the warp
// has signalled a barrier, an MMA issued after waiting on it reads the rotated values.
// Rotates two tiles whose rows sit at the same positions (an item's Q and K tiles): rows
// [0, ra) of tile_a and [0, rb) of tile_b (rb may be 0), row r at position pos0 + r,
// shared among nw rotating warps.  A lane keeps one 16-byte chunk (four column pairs)
// and walks the rows 32 / (D/8) apart; it loads the (cos, sin) of its pairs once, for its
// first row and for the step between its rows, and advances them by the angle-addition
// formulas (cos(x+d) = cos x cos d - sin x sin d, sin(x+d) = sin x cos d + cos x sin d), so
// that no table load waits inside the loop.  A warp's share is a few rows, so a lane takes
// a few steps (up to 8 at D = 128 with eight warps): the recurrence adds about 1e-7
// relative error per step, far below the bf16 rounding of the rotated values.
__device__ __forceinline__ float4 rope_advance(float4 cs, float4 st) {
  return make_float4(fmaf(cs.x, st.x, -cs.y * st.y), fmaf(cs.y, st.x, cs.x * st.y),
                     fmaf(cs.z, st.z, -cs.w * st.w), fmaf(cs.w, st.z, cs.z * st.w));
}
template <int D>
__device__ __forceinline__ void rope_rotate_pair_share(uint32_t tile_a, int ra, uint32_t tile_b, int rb,
                                                       int pos0, const float2* __restrict__ table, int wi,
                                                       int nw, int lane) {
  constexpr int kChunks = D / 8;          // 16-byte chunks per row
  constexpr int kRowsPer = 32 / kChunks;  // rows a warp covers per pass
  static_assert(kChunks <= 32 && 32 % kChunks == 0, "a warp covers whole rows");
  const int rows = max(ra, rb);
  const int per = (rows + nw - 1) / nw;
  const int r0 = min(rows, wi * per), r1 = min(rows, r0 + per);
  const int cc = lane % kChunks, a = cc >> 3, c = cc & 7;
  int r = r0 + lane / kChunks;
  if (r < r1) {
    const float4* tb = reinterpret_cast<const float4*>(table + (size_t)(pos0 + r) * (D / 2) + a * 32 + c * 4);
    const float4* ts = reinterpret_cast<const float4*>(table + (size_t)kRowsPer * (D / 2) + a * 32 + c * 4);
    float4 c01 = __ldg(tb), c23 = __ldg(tb + 1);
    const float4 s01 = __ldg(ts), s23 = __ldg(ts + 1);
    for (; r < r1; r += kRowsPer) {
      const uint32_t off = a * 16384u + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
      if (r < ra) {
        uint4 v = ld_shared_v4(tile_a + off);
        v.x = rope_rotate_word(v.x, c01.x, c01.y);
        v.y = rope_rotate_word(v.y, c01.z, c01.w);
        v.z = rope_rotate_word(v.z, c23.x, c23.y);
        v.w = rope_rotate_word(v.w, c23.z, c23.w);
        st_shared_v4(tile_a + off, v.x, v.y, v.z, v.w);
      }
      if (r < rb) {
        uint4 v = ld_shared_v4(tile_b + off);
        v.x = rope_rotate_word(v.x, c01.x, c01.y);
        v.y = rope_rotate_word(v.y, c01.z, c01.w);
        v.z = rope_rotate_word(v.z, c23.x, c23.y);
        v.w = rope_rotate_word(v.w, c23.z, c23.w);
        st_shared_v4(tile_b + off, v.x, v.y, v.z, v.w);
      }
      c01 = rope_advance(c01, s01);
      c23 = rope_advance(c23, s23);
    }
  }
  fence_proxy_async_smem();
}

// Rows of a 128-row tile starting at position pos0 that the rotation covers: the rows of
// the sequence (len rows) that the table has positions for (npos).
__device__ __forceinline__ int rope_rows(int pos0, int len, int npos) {
  return max(0, min(128, min(len, npos) - pos0));
}

// The transpose of the rotation on n consecutive fp32 columns of one row (a gradient with
// respect to rotated values back to the unrotated ones): columns col0 + 2t, col0 + 2t + 1
// form the pair i = col0/2 + t, turned by the angle of position pos backwards.
template <int N>
__device__ __forceinline__ void rope_unrotate_row(float* x, int col0, int pos, int D,
                                                  const float2* __restrict__ table) {
  const float2* tb = table + (size_t)pos * (D / 2) + col0 / 2;
#pragma unroll
  for (int t = 0; t < N / 2; ++t) {
    const float2 cs = __ldg(tb + t);
    const float y0 = x[2 * t], y1 = x[2 * t + 1];
    x[2 * t] = fmaf(y0, cs.x, y1 * cs.y);
    x[2 * t + 1] = fmaf(y1, cs.x, -y0 * cs.y);
  }
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a stack of
// 128-byte-swizzled atoms (8 rows x 128 bytes per atom).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace tc
}  // namespace jfa
