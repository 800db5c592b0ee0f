// Shared device utilities and kernel-argument structs of the draft-tree library.
// sm_103a only: tcgen05 / TMA / mbarrier through inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define EAGLE_DEV __device__ __forceinline__
#define EAGLE_MAX_DEPTH_INTERNAL 16

namespace eagle {

// ------------------------------------------------------------------ constants
constexpr int BM = 128;            // GEMM tile: output features per tile (TMEM lanes)
constexpr int BK = 64;             // GEMM tile: K per pipeline stage (one 128-byte swizzle row)
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int MAX_ROWS_PER_BLOCK = 128;   // rows of one row block (hi+lo = 256 MMA columns)
constexpr int KMAX = 16;                  // max children per node
constexpr int ATT_CHUNK = 64;             // prefix keys per attention split
constexpr long long WAIT_LIMIT_CYCLES = 2000000000LL;   // ~1 s at 2 GHz

constexpr unsigned DEVERR_TIMEOUT = 0x1u;
constexpr unsigned DEVERR_PREFIX = 0x2u;
constexpr unsigned DEVERR_TOKEN = 0x4u;
constexpr unsigned DEVERR_SELECT = 0x8u;

// ---------------------------------------------------------- small helpers
EAGLE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

EAGLE_DEV float bf16_to_f32(uint16_t u) { return __uint_as_float(static_cast<uint32_t>(u) << 16); }

// round-to-nearest-even float -> bf16 bits (hardware conversion)
EAGLE_DEV uint16_t f32_to_bf16(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

// hi / lo parts (as above) of two floats, each pair packed with the first float in the low
// half: one packed round-to-nearest-even conversion for the two hi parts, one for the lo parts
EAGLE_DEV void split2_packed(float x, float y, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(y), "f"(x));
  const float hx = __uint_as_float(hi << 16), hy = __uint_as_float(hi & 0xFFFF0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(y - hy), "f"(x - hx));
}
// 2^x on the special-function unit (relative error ~2^-22; 2^-inf = 0)
EAGLE_DEV float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): ~16 significant bits in two bf16s
EAGLE_DEV void split_hilo(float x, uint16_t& hi, uint16_t& lo) {
  hi = f32_to_bf16(x);
  lo = f32_to_bf16(x - bf16_to_f32(hi));
}

EAGLE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
EAGLE_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// a value as the rankings see it: NaN ranks below everything, so a ranking stays a strict
// order (exactly the requested number of winners) whatever the inputs hold
EAGLE_DEV float rank_value(float v) { return v != v ? -INFINITY : v; }

// total order used for every top-k of this library: larger value first, then smaller id
EAGLE_DEV bool beats(float v, int id, float w, int wid) {
  return v > w || (v == w && id < wid);
}

// ------------------------------------------------ counter-based random numbers
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC 2011): each round multiplies counter words 0 and 2 by the two round
// constants, XORs the high halves of the products with the other two words and the key,
// and permutes; the key advances by the two Weyl constants between rounds.
EAGLE_DEV uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}
// Gumbel noise -log(-log U) of a 32-bit word x, U = (x + 1/2) / 2^32: -log U is taken
// from U itself below 1/2 and as -log1p(-(1 - U)) above, 1 - U = (2^32 - 1 - x + 1/2) / 2^32
// formed from the exact integer, so that neither end loses its precision.
EAGLE_DEV float gumbel_of_word(uint32_t x) {
  const float e = x < 0x80000000u ? -logf((static_cast<float>(x) + 0.5f) * 2.3283064365386963e-10f)
                                  : -log1pf(-(static_cast<float>(0xFFFFFFFFu - x) + 0.5f) * 2.3283064365386963e-10f);
  return -logf(e);
}
// The Gumbel noise of token t of row i at depth s under a request's 64-bit seed: word
// (t mod 128) / 32 of Philox(counter = (32 (t / 128) + t mod 32, i, s, 0), key = seed).
EAGLE_DEV float token_gumbel(int t, int i, int s, unsigned long long seed) {
  const uint4 w = philox4x32_10(make_uint4(32u * static_cast<uint32_t>(t >> 7) + (t & 31), static_cast<uint32_t>(i),
                                           static_cast<uint32_t>(s), 0u),
                                static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const int j = (t & 127) >> 5;
  return gumbel_of_word(j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w);
}

// named barrier among `nthreads` threads (id 1.. ; 0 is __syncthreads)
EAGLE_DEV void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// named barrier that also returns whether `pred` held in any of the `nthreads` threads
EAGLE_DEV bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// programmatic dependent launch
EAGLE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
EAGLE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
EAGLE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
EAGLE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
EAGLE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
EAGLE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns false (and
// sets DEVERR_TIMEOUT in *err and the CTA-wide abort flag) when the limit runs out or
// another role of the CTA already aborted.
EAGLE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag,
                         long long limit = WAIT_LIMIT_CYCLES) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) {
        atomicOr(err, DEVERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// The same wait for roles that can afford to wake up late: after a few polls the thread
// sleeps between polls, so a waiting warp neither takes issue slots from its neighbours on the
// SM sub-partition nor hammers the barrier's shared-memory bank.
EAGLE_DEV bool mbar_wait_sleepy(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag,
                                long long limit = WAIT_LIMIT_CYCLES) {
  for (int i = 0; i < 4; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) {
        atomicOr(err, DEVERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}
EAGLE_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
EAGLE_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// --------------------------------------------------------------------- TMA
EAGLE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
EAGLE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
EAGLE_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar,
                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
// the same tile into the shared memory of every CTA of the cluster in cta_mask (same offset),
// completing the bytes on the mbarrier at the same offset in each
EAGLE_DEV void tma_load_2d_mc(uint32_t dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar, uint64_t policy,
                              uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar), "h"(cta_mask), "l"(policy)
      : "memory");
}
EAGLE_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, uint32_t bar,
                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}
// the same box into L2 only (no shared memory, no barrier)
EAGLE_DEV void tma_prefetch_l2_3d(const CUtensorMap* tm, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(reinterpret_cast<uint64_t>(tm)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
EAGLE_DEV void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// ----------------------------------------------------------------- tcgen05
EAGLE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
EAGLE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
EAGLE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
EAGLE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
EAGLE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, f32 accumulate
EAGLE_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A's rows in the TMEM lanes, its K elements packed two
// bf16 to a 32-bit column (first element in the low half)
EAGLE_DEV void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 consecutive 32-bit columns of this warp's 32 TMEM lanes, to / from registers
EAGLE_DEV void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
EAGLE_DEV void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// arrive on `bar` once every tcgen05 op issued so far by this thread has completed
EAGLE_DEV void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// arrive on the mbarrier at offset `bar` of every CTA in cta_mask once this thread's
// tcgen05 ops so far have completed
EAGLE_DEV void tc_commit_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes
EAGLE_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
EAGLE_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes, from registers
EAGLE_DEV void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
EAGLE_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout that
// TMA's SWIZZLE_128B writes (rows of 128 bytes, 8-row atoms of 1024 bytes).
EAGLE_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
  d |= static_cast<uint64_t>(1) << 16;                     // leading byte offset (unused for SW128 K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;             // stride byte offset: next 8-row atom
  d |= static_cast<uint64_t>(1) << 46;                     // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                     // layout: 128-byte swizzle
  return d;
}
// The same for an MN-major operand (the MN index runs along the 128-byte rows): 64-element
// groups of the MN dimension `lbo` bytes apart, 8-row groups of the K dimension `sbo` apart.
EAGLE_DEV uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, f32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled tile
EAGLE_DEV uint32_t sw128_offset(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// ------------------------------------------------------- GEMM argument structs
// How the GEMM's activation operand (rows x K) is formed from global memory.
enum BMode : int {
  B_F32 = 0,      // x[row][k] f32
  B_NORM = 1,     // RMSNorm: x[row][k] * rstd[row] * gamma[k], rstd from sum-of-squares partials
  B_FC = 2,       // [feat(row_feat[row]) ; emb(row_tok[row])]: K = 2 * split
  B_SWIGLU = 3,   // silu(x[row][k]) * x[row][split + k] (gate | up halves)
  B_BF16 = 4,     // x[row][k] bf16
  B_TMA = 5       // tile loaded by TMA from an operand copy: bf16 rows 2r = hi(x_r), 2r+1 = lo(x_r)
};

struct BSrc {
  int mode;
  const float* x;          // B_F32 / B_NORM / B_SWIGLU / B_FC (feature rows)
  int ldx;                 // row stride (elements)
  const uint16_t* xb;      // B_BF16
  // B_NORM
  const float* ss;         // [ss_tiles][ss_ld] partial sums of squares
  int ss_tiles, ss_ld;
  const float* gamma;
  float eps;
  int dnorm;
  // B_FC / B_SWIGLU
  int split;               // B_FC: d (feature part width); B_SWIGLU: d_ff
  const int* row_feat;     // B_FC: feature row of each GEMM row
  const int* row_tok;      // B_FC: token of each GEMM row
  const void* emb;         // B_FC: embedding table [vocab][split]
  int emb_bf16;
};

enum EpiKind : int { EPI_STORE = 0, EPI_QKV = 1, EPI_LMHEAD = 2, EPI_SWIGLU = 3, EPI_LOGITS = 4 };

struct EpiArgs {
  int kind;
  // EPI_STORE: out[row][m] = acc (+ resid[row][m]); ss[tile][row] = sum over the tile of out^2
  float* out;
  int ldo;
  const float* resid;
  int ldr;
  float* ss;
  int ss_ld;
  // EPI_QKV: rotary embedding, queries to q, keys/values to the tree KV rows
  float* q;
  float* tk;
  float* tv;
  const int* row_req;      // request of each GEMM row
  const int* row_slot;     // request-local tree row
  const int* row_pos;      // position id
  const float* rope_cos;   // [max_pos][hd/2]
  const float* rope_sin;
  int max_pos;
  int Hq, Hkv, hd, tree_rows;
  // EPI_LMHEAD: per vocabulary tile and row: max and sum of exp; per CTA and row: top-k
  float* lm_max;           // [N][tiles]
  float* lm_sum;           // [N][tiles]
  float* lm_val;           // [N][grid][k]  (each row's CTA lists contiguous)
  int* lm_id;              // [N][grid][k]
  int topk;
  // sampled drafting (EPI_LMHEAD, seeds != null): the top-k is taken over logit + Gumbel
  // noise of (request, frontier slot, depth) = (row / sample_rows, row % sample_rows,
  // sample_depth), row = sample_row0 + the launch's row; the log-sum-exp stays unperturbed
  const unsigned long long* seeds;
  int sample_rows, sample_depth, sample_row0;
  float* logits;           // EPI_LOGITS, or EPI_LMHEAD (nullable): the rows' full logits [N][M]
                           // (after the factored norm)
  // operand copy for the next GEMM (EPI_STORE, EPI_SWIGLU):
  // hl[2 row][m] = hi, hl[2 row + 1][m] = lo of value * hl_gamma[m] (hl_gamma may be null)
  uint16_t* hl;
  int hl_ld;
  const float* hl_gamma;
  // factored RMSNorm of the operand (EPI_QKV, EPI_SWIGLU): acc[row] *= 1/sqrt(mean + eps),
  // mean from the producer's per-tile sums of squares nss[tile][row]
  const float* nss;
  int nss_tiles, nss_ld, nss_d;
  float nss_eps;
};

struct GemmArgs {
  int M, K, N;             // N = rows
  int MT, KB;              // tiles of M (per weight map), K blocks
  int m_split;             // rows [0, m_split) from weight map 0, [m_split, M) from map 1
  int a_pair;              // tile = 64 rows of map 0 + the same 64 rows of map 1 (gate | up)
  int b_tma;               // activation tile by TMA (operand copy) instead of the converter warps
  int npad;                // padded rows per row block (multiple of 16)
  int nrb;                 // row blocks
  int tmem_cols;           // allocated TMEM columns
  int nbuf;                // accumulator buffers in TMEM (2 = epilogue overlaps next unit)
  int stages;
  int kpair;               // 1: two consecutive K blocks per pipeline stage (TMA operand only),
                           // so one barrier round trip and one issue loop pass cover 8 MMAs
  int csplit;              // 0: stream-K over (tile, K block) units; S >= 1: S CTAs per tile (a
                           // cluster when S > 1) on consecutive K ranges, reduced through DSMEM
  BSrc b;
  EpiArgs e;
  long long wait_limit;    // clock cycles a bounded wait may take (0: the default, ~1 s)
  float* part;             // split-K partial scratch [grid][2][nrb*npad][BM]
  int* counters;           // per tile arrival counters (zero between launches)
  unsigned* err;
};

}  // namespace eagle
