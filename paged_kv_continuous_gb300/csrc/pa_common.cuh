// Device-side building blocks shared by the kernels of libpa_gb300.so:
// mbarrier and bulk-copy (TMA) wrappers in inline PTX for sm_103a, bounded
// pipeline waits, bf16 unpacking and the device error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pa.h"

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
// A pipeline wait gives up after this many SM clock cycles (about 2 s at
// 2 GHz, longer at lower clocks), ORs PA_DEVERR_WAIT_TIMEOUT into the error
// word and lets the kernel run out without touching memory again.
constexpr long long kWaitTimeoutCycles = 4000000000ll;

// Programmatic dependent launch.  A kernel launched with it may begin while
// the previous kernel in the stream is still running; griddep_wait() returns
// once that kernel has completed and its memory is visible, and
// griddep_launch_dependents() lets the next such kernel begin early.  Both
// are no-ops in a kernel launched without the attribute.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel`, with programmatic dependent launch when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises `kernel`'s dynamic shared memory limit to `bytes` the first time it
// is launched on `device` (one flag per device; devices past the table are
// set every time).  The flags are atomic: several host threads may call on
// one device at once, and setting the attribute twice is harmless.
template <typename Kernel>
cudaError_t set_smem_once(std::atomic<bool> (&done)[64], Kernel kernel, int device, int bytes) {
  const bool tracked = device >= 0 && device < 64;
  if (tracked && done[device].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) done[device].store(true, std::memory_order_release);
  return e;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void report(int32_t *err, int bits) {
  if (err) atomicOr(err, bits);
}

// ---- mbarrier ------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Adds `bytes` to the barrier's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of phase `parity` (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of the barrier.  Gives up when *abort is set (by
// another warp that already gave up) or after kWaitTimeoutCycles SM cycles;
// in the latter case it sets *abort and reports PA_DEVERR_WAIT_TIMEOUT.
// Returns true when the phase completed.  The time limit uses the SM cycle
// counter (a register read); a few waits are tried before it is read at all.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int32_t *err) {
#pragma unroll 1
  for (int i = 0; i < 4; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      *abort = 1;
      report(err, PA_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---- bulk copies (TMA, non-tensor) ---------------------------------------

// Global -> shared bulk copy completing on an mbarrier.  dst, src and bytes
// must be multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policies for bulk loads: KV pages are streamed once per step, the small
// per-sequence rows (q) are kept.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- named barrier among a subset of warps --------------------------------

// Non-aligned form: lanes of a warp may arrive from divergent paths.
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- bf16 helpers --------------------------------------------------------

// Two bf16 values packed in a 32-bit word (element 0 in the low half) to
// fp32: a bf16 is the high half of an fp32, so both widenings are exact.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// fp32 -> bf16 with round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Rotate-half RoPE of 8 bf16 pairs: a holds dims d .. d + 7 of a head row, b
// their partners d + 64 .. d + 71; c0 / c1 and s0 / s1 the cos and sin table
// entries of dims d .. d + 7.  ra = a c - b s, rb = b c + a s, each element
// one fused multiply-add over a rounded product, then one rounding to bf16.
// The store kernel with RoPE and the fused decode step both rotate with it,
// so their rotated rows are the same bits.
__device__ __forceinline__ void rope_rotate8(const uint4 &a, const uint4 &b, const float4 &c0,
                                             const float4 &c1, const float4 &s0,
                                             const float4 &s1, uint4 &ra, uint4 &rb) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
  const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t ow[4], pw[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 x1 = bf16x2_to_float2(aw[w]), x2 = bf16x2_to_float2(bw[w]);
    const float c_lo = cs[2 * w], c_hi = cs[2 * w + 1];
    const float s_lo = sn[2 * w], s_hi = sn[2 * w + 1];
    ow[w] = float2_to_bf16x2(fmaf(x1.x, c_lo, -(x2.x * s_lo)), fmaf(x1.y, c_hi, -(x2.y * s_hi)));
    pw[w] = float2_to_bf16x2(fmaf(x2.x, c_lo, x1.x * s_lo), fmaf(x2.y, c_hi, x1.y * s_hi));
  }
  ra = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  rb = make_uint4(pw[0], pw[1], pw[2], pw[3]);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ int ceil_div_blocks(int n) { return (n + kBlockSize - 1) / kBlockSize; }

// Decode split partition.  Split c of S over N global blocks starts at
// floor(N W(c) / W(S)), W(c) the summed weights of splits 0 .. c - 1.
// Every split weighs 4, except that with S >= 32 and N >= 4 S the last four
// weigh 3, 3, 3 and 2: in a chain of launches the hardware starts a grid's
// CTAs in index order, so the highest-indexed ones land on the SMs the
// previous kernel frees last and start up to a few microseconds after the
// rest; a lighter share lets them end with the others (the rest take under
// one percent more).  With N >= 4 S even the lightest split holds at least
// two blocks, so N >= S still means that every split holds a block.
__device__ __forceinline__ bool split_light_tail(long long S, long long N) {
  return S >= 32 && N >= 4 * S;
}
__device__ __forceinline__ long long split_weight_before(long long c, long long S) {
  const long long base = S - 4;
  if (c <= base) return 4 * c;
  const long long t = c - base;  // 1 .. 4
  return 4 * base + (t == 1 ? 3 : t == 2 ? 6 : t == 3 ? 9 : 11);
}
__device__ __forceinline__ long long split_begin(long long c, long long S, long long N) {
  if (!split_light_tail(S, N)) return c * N / S;
  return N * split_weight_before(c, S) / split_weight_before(S, S);
}
// The split holding global block x: the largest c with split_begin(c) <= x,
// i.e. the largest c with W(c) <= floor(((x + 1) W(S) - 1) / N).
__device__ __forceinline__ long long split_of_block(long long x, long long S, long long N) {
  if (!split_light_tail(S, N)) return ((x + 1) * S - 1) / N;
  const long long v = ((x + 1) * split_weight_before(S, S) - 1) / N;
  const long long b4 = 4 * (S - 4);
  if (v < b4 + 3) return v / 4 < S - 4 ? v / 4 : S - 4;
  if (v < b4 + 6) return S - 3;
  if (v < b4 + 9) return S - 2;
  return S - 1;
}

}  // namespace pa
