// plmla_decode_tc.cu -- split-KV gated-MLA decode on the 5th-generation tensor
// cores (tcgen05 + TMEM) with TMA page loads, for sm_103a.
//
// What one CTA computes: the partial softmax state of one KV chunk [t0, t1) of
// one request for NG query rows (draft token j, head h):
//   o_part = sum_t softmax(s)_t c_t over the chunk,   lse_part = ln sum_t e^{s_t}
// with s_t = scale * (q_nope_absorbed . c_t + q_rope . k_rope_t), all rows
// sharing the chunk's latent rows (absorbed MLA: TokenSpeed Kimi K3 post,
// architecture list; chunks and their merge: its "Gluon kernels on AMD GPUs"
// section, and the AgentX post's per-request splitting).
//
// Layout of the work (the "transposed" form, so that every MMA is M = 128 and
// uses the one-row-per-TMEM-lane accumulator layout):
//   S^T[t, r]  = K_tile[t, 0:576] . Q[r, 0:576]      M = 128 tokens, N = NG rows
//   O^T[l, r] += V_tile^T[l, t] . P^T[t, r]          M = 128 latent (x4), N = NG
// A = the KV tile in shared memory (K-major for S^T, MN-major for O^T: the same
// bytes), B = Q^T (K-major) or P^T (MN-major).  TMEM holds O^T in four 128-lane
// blocks (columns 0..255) and S^T at columns 256..256+NG.
//
// KV tiles are 128 tokens (always inside one 1,536-token page) read from a 3-D
// tensor map [page][token][576] over the slab: page IDs come from the page
// table with the table's row stride, and the page offset is 64-bit inside the
// TMA unit (pools above 2 GB; AgentX - InferenceXv3 report, ROCm AITER section).
// Shared memory holds Q^T (bf16: 9 x NG x 128 B), the probability tile P^T,
// and two rings of 16 KB slots through which every tile streams twice:
//   K ring: the nine 128 x 64 column blocks of the tile, for S^T (from HBM);
//   V ring: eight 64-token x 128-latent blocks of the same tile, for O^T
//           (a re-read that hits L2), each covering both 64-column halves of
//           one 128-row O^T block.
// (E4M3 pages: see Fmt below.)
// S^T and P^T V are issued by two threads in different warps: at M = 128,
// N <= 64 a single issuing thread cannot keep the tensor pipe busy.  S^T is
// double-buffered in TMEM, so S^T of tile i+1 runs while the softmax of tile i
// does, and each ring is consumed in order by its own issuer.
//
// Warp roles (384 threads): warp 0 = K/Q producer, warp 1 = S^T issuer and
// TMEM owner, warps 2..9 = softmax (two warps per TMEM lane quadrant, each with
// half of a token's query-row columns; the same threads write the partial
// output, one thread per latent row of O^T and column half), warp 10 = V
// producer, warp 11 = P^T V issuer.
// Two softmax warps per SM sub-partition keep the dependent softmax arithmetic
// from exposing its full latency.
//
// Online softmax in fp32 with a lagged maximum: the reference maximum m of a
// row moves only when a score exceeds it by more than kTau (log2 units).  Each
// tile, every token lane tests its scores against m and one barrier ORs the
// answers; only then (always on a segment's first tile, rarely after) are the
// column maxima reduced across the 128 lanes (warp shuffles + shared memory)
// and O^T's columns and the running sums rescaled.  P = 2^(s*scale*log2e - m)
// <= 2^kTau stays finite in bf16.
//
// Tokens at or past the chunk end (the request's last, partial tile) are
// masked in the scores (probability 0), and the V producer loads only the
// item rows inside the history: the slot rows past it keep what the slot held
// before, zeros written at kernel start or earlier history rows, finite either
// way, so stale or NaN page contents never reach the output (0 * NaN would).
//
// Teams in clusters (CL = 2 or 4, bf16 pages): the CTAs of CL teams of one
// member, which stream the same KV items, run as one thread-block cluster.  Item
// n of each ring is loaded by the CTA of rank n % CL with a TMA multicast into
// the same slot of every CTA (each CTA's own producer posts the expected bytes
// on its own full barrier), and every MMA thread releases a slot with a
// multicast commit to the empty barrier of every CTA, which thus counts CL
// releases.  Cluster barriers after initialisation and before exit keep every
// remote write inside the lifetime of its target.  Only the loads change, never
// the arithmetic.
//
// Every mbarrier wait is bounded: after kWaitLimitNs the waiting thread sets
// the workspace status word and a CTA-wide abort flag, the producer waits (with
// its own bound) for the copies it issued, each MMA thread waits for its MMAs,
// and TMEM is freed before the CTA exits.
#include <cuda.h>
#include <math.h>

#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = 8;                // warps 2..9: two per TMEM lane quadrant
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kWarpVProducer = 10, kWarpPvIssuer = 11;
constexpr int kSubBytes = kTile * 64 * 2;       // one ring slot: 16 KB
constexpr int kVHalf = 64 * 64 * 2;             // one 64 x 64 half of a bf16 V item
constexpr int kTmemCols = 512;
constexpr int kTmemS = 256;                     // S^T buffers from column 256 on
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
constexpr int kMaxDynSmem = 232448;
constexpr int kMaxK = 8, kMaxV = 8;             // ring slots (K, V) at most

// How a 128-token tile moves through the rings, per cache format.
//   bf16 pages: nine K items of 64 columns (8 latent blocks + the rope block),
//     4 MMAs of K = 16 each; eight V items of 64 tokens x 128 latent rows, each
//     two 64-column TMA boxes; P^T in bf16 (tcgen05 kind::f16).
//   E4M3 pages (FP8 cache): five K items of 128 byte-columns (4 latent blocks +
//     the rope block, whose upper 64 columns the TMA unit fills with zeros and no
//     MMA reads), 4 MMAs of K = 32 each (2 on the rope) with N = 2 NG: the B
//     operand stacks the hi rows of the two-part query over its lo rows, so the
//     K tile is read once and S^T holds hi and lo scores side by side (the
//     softmax adds them); four V items of 128 tokens x 128 latent rows; P^T in
//     E4M3 (kind::f8f6f4, E4M3 x E4M3).
// P = 2^(x - m + p_off) with x - m <= tau keeps P finite in its format; the
// E4M3 offset moves the bulk of a diffuse softmax above E4M3's subnormals.
template <bool F8>
struct Fmt {
    static constexpr int sub = F8 ? 5 : 9;              // K items per tile
    static constexpr int col_step = F8 ? 128 : 64;      // K item width (elements)
    static constexpr int rope_mmas = F8 ? 2 : 4;        // MMAs on the rope item
    static constexpr int v_tokens = F8 ? 128 : 64;      // tokens per V item
    static constexpr int s_rows = F8 ? 2 : 1;           // S^T columns per query row (hi, lo)
    static constexpr int s_stride = F8 ? 128 : 64;      // TMEM columns between S^T buffers
    static constexpr int v_per_block = kTile / v_tokens; // V items per 128-latent block
    static constexpr int v_items = 4 * v_per_block;     // V items per tile
    static constexpr int v_slot = v_tokens * 128 * (F8 ? 1 : 2);   // bytes per V item (ring slot)
    static constexpr float tau = F8 ? 4.f : 8.f;        // lagged-maximum threshold (log2)
    static constexpr float p_off = F8 ? 4.f : 0.f;
};

template <int NG, bool F8>
struct Smem {
    using F = Fmt<F8>;
    static constexpr int pn = F8 && NG < 32 ? 32 : NG;      // P^T columns (MMA N of P^T V)
    static constexpr int p_row = F8 ? pn : 2 * NG;          // bytes per token row of P^T
    // Q^T: bf16 nine 128-byte column blocks of NG rows; E4M3 four 128-byte latent
    // blocks and the rope block of 64 bytes per row (64-byte swizzle), each with
    // the NG hi rows of the two-part query followed by its NG lo rows
    static constexpr int q_chunk = F::s_rows * NG * 128;    // one 128-byte column block
    static constexpr int q_lo = NG * 128;                   // lo rows within a block (E4M3)
    static constexpr int q_rope_bytes = F8 ? 2 * NG * 64 : q_chunk;
    static constexpr int q_rope_lo = NG * 64;               // lo rows within the rope block
    static constexpr int q_bytes = (F::sub - 1) * q_chunk + q_rope_bytes;
    static constexpr int p_bytes = kTile * p_row;           // P^T
    static constexpr int bar_bytes = 512;
    static constexpr int misc_bytes = bar_bytes + 4 * 64 * 4 + 4 * 64 * 4 + 32;
    // no alignment slack: the dynamic shared memory base is 1024-aligned (the
    // kernel checks it on entry)
    static constexpr int fixed = p_bytes + q_bytes + misc_bytes;
    static constexpr int avail = kMaxDynSmem - fixed;
    // bf16: half of the 16 KB slots for each ring; E4M3: four 8 KB V slots (half
    // a tile), the rest K
    static constexpr int v_slots = F8 ? 4 : ((avail / kSubBytes) / 2 < kMaxV ? (avail / kSubBytes) / 2 : kMaxV);
    static constexpr int k_fit = (avail - v_slots * F::v_slot) / kSubBytes;
    static constexpr int k_slots = k_fit < kMaxK ? k_fit : kMaxK;
    static constexpr int v_off = k_slots * kSubBytes;
    static constexpr int p_off = v_off + v_slots * F::v_slot;
    static constexpr int q_off = p_off + p_bytes;            // 1024-aligned
    static constexpr int bar_off = q_off + q_bytes;          // 1024-aligned
    static constexpr int red_off = bar_off + bar_bytes;      // float red[4][64]
    static constexpr int fin_off = red_off + 4 * 64 * 4;     // float fin[64]
    static constexpr int m_off = fin_off + 64 * 4;           // float m[64]   (log2 units)
    static constexpr int al_off = m_off + 64 * 4;            // float alpha[64]
    static constexpr int cf_off = al_off + 64 * 4;           // float cf[64]  (E4M3 score factors)
    static constexpr int misc_off = cf_off + 64 * 4;         // tmem addr, abort, need[2]
    static constexpr int bytes = misc_off + 32;
    static constexpr int alloc = bytes;
    static_assert(k_slots >= 2 && v_slots >= 2, "ring depth");
    static_assert(p_bytes % 1024 == 0 && q_chunk % 1024 == 0 && q_lo % 1024 == 0 &&
                      q_rope_lo % 512 == 0 && F::v_slot % 1024 == 0 && F::s_rows * NG <= F::s_stride,
                  "swizzle atom alignment");
    static_assert(alloc <= kMaxDynSmem, "shared memory budget");
};

// barrier offsets inside the barrier area (8 bytes each)
constexpr int kBarFullK = 0, kBarEmptyK = 64, kBarFullV = 128, kBarEmptyV = 192;
constexpr int kBarQ = 264, kBarQe = 272, kBarS = 280, kBarSfree = 296;
constexpr int kBarP = 312, kBarPv = 320, kBarOf = 328, kBarDrainS = 336, kBarDrainPv = 344;
constexpr int kBarPvIssued = 352;                // [4] P^T V of tile g issued, on barrier g % 4
// S^T of tile g waits until P^T V of tile g - lead has been issued (lead <= 3,
// so that the next phase of that barrier, tile g - lead + 4, cannot complete
// first): two tiles for bf16 pages, three for E4M3 pages, whose tiles are half
// the bytes (measured best for each).
template <bool F8>
constexpr int kLead = F8 ? 3 : 2;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Slow path of wait_bounded.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       int32_t *status, int32_t code)
{
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag)
                return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicExch(status, code);
                return false;
            }
        }
    }
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when another thread of the CTA aborted, or after
// kWaitLimitNs, in which case it raises the abort flag and the status word.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int *abort_flag, int32_t *status,
                                             int32_t code)
{
    return mbar_try_wait(bar, parity) || wait_slow(bar, parity, abort_flag, status, code);
}

// Wait used while tearing down: only time-bounded.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kDrainLimitNs)
            return;
    }
}

// A 3-D tiled TMA load into shared memory, completing on an mbarrier, with an
// L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                                 int c2, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// The hinted load delivered to the same shared-memory offset of every CTA in
// `cta_mask` (thread-block cluster), completing on the barrier at the same
// offset in each of them.
__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                               int c2, uint32_t bar, uint16_t cta_mask,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6, %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "h"(cta_mask),
        "l"(policy)
        : "memory");
}

// A KV load into the ring slot at `dst`: to this CTA alone (CL = 1) or to all
// CL CTAs of the cluster.
template <int CL>
__device__ __forceinline__ void kv_load(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                        uint32_t bar, uint64_t policy)
{
    if constexpr (CL == 1)
        tma_load_3d_hint(dst, map, c0, c1, c2, bar, policy);
    else
        tma_load_3d_mc(dst, map, c0, c1, c2, bar, (uint16_t)((1u << CL) - 1u), policy);
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Prefetch one box of a tiled tensor into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start, leading/stride byte offsets
// (16-byte units), descriptor version 1, swizzle layout in bits 61..63.
constexpr uint32_t kSw128 = 2, kSw64 = 4, kSw32 = 6;

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout)
{
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4: fp32 accumulate, E4M3 A and B.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

template <bool F8>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                    uint32_t accumulate)
{
    if constexpr (F8)
        mma_e4m3(d_tmem, a, b, idesc, accumulate);
    else
        mma_bf16(d_tmem, a, b, idesc, accumulate);
}

template <bool F8>
__host__ __device__ constexpr uint32_t idesc_for(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return F8 ? idesc_e4m3(M, N, a_mn_major, b_mn_major)
              : idesc_bf16(M, N, a_mn_major, b_mn_major);
}

// Swizzle mode of a K- or MN-major operand whose rows are `row_bytes` wide.
__host__ __device__ constexpr uint32_t layout_for_row(int row_bytes)
{
    return row_bytes == 128 ? kSw128 : (row_bytes == 64 ? kSw64 : kSw32);
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Arrive on the barrier at offset `bar` of every CTA of the cluster once this
// thread's MMAs so far have completed (CL = 1: this CTA's barrier).
template <int CL>
__device__ __forceinline__ void mma_commit_all(uint32_t bar)
{
    if constexpr (CL == 1) {
        mma_commit(bar);
    } else {
        const uint16_t mask = (uint16_t)((1u << CL) - 1u);
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
            "h"(mask)
            : "memory");
    }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Load C consecutive fp32 TMEM columns of this thread's lane (C = 8, 16 or 32).
template <int C>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&v)[C])
{
    if constexpr (C % 16 == 0) {
#pragma unroll
        for (int b = 0; b < C / 16; ++b) {
            uint32_t r[16];
            tmem_ld16(taddr + 16 * b, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e)
                v[16 * b + e] = __uint_as_float(r[e]);
        }
    } else {
        static_assert(C == 8, "column count");
        uint32_t r[8];
        tmem_ld8(taddr, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e)
            v[e] = __uint_as_float(r[e]);
    }
}

// Multiply C consecutive fp32 TMEM columns of this thread's lane by alpha[col].
template <int C>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, uint32_t alpha_addr)
{
    if constexpr (C % 16 == 0) {
#pragma unroll
        for (int b = 0; b < C / 16; ++b) {
            uint32_t r[16];
            tmem_ld16(taddr + 16 * b, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float al;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(al) : "r"(alpha_addr + 4 * (16 * b + e)));
                r[e] = __float_as_uint(__uint_as_float(r[e]) * al);
            }
            tmem_st16(taddr + 16 * b, r);
        }
    } else {
        static_assert(C == 8, "column count");
        uint32_t r[8];
        tmem_ld8(taddr, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float al;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(al) : "r"(alpha_addr + 4 * e));
            r[e] = __float_as_uint(__uint_as_float(r[e]) * al);
        }
        tmem_st8(taddr, r);
    }
}


__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Named barrier over the 128 softmax threads that also ORs a predicate: every
// thread gets the same answer, so an abort decided here is taken uniformly.
__device__ __forceinline__ bool softmax_bar_or(bool pred)
{
    uint32_t res;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 256, q;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(res)
        : "r"(pred ? 1u : 0u)
        : "memory");
    return res != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Butterfly reduce-scatter of NG per-lane values across a warp.  Afterwards
// lane l holds the warp-wide result for columns [l*NG/32, (l+1)*NG/32) when
// NG >= 32, or for column l / (32/NG) when NG < 32.
template <int NG, bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[NG], int lane)
{
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        const int o = 16 >> st;
        const int half = NG >> (st + 1);
        if (half >= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float lo = v[i], hi = v[i + half];
                const float send = upper ? lo : hi;
                const float keep = upper ? hi : lo;
                const float recv = __shfl_xor_sync(0xffffffffu, send, o);
                v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
            }
        } else {
            const float recv = __shfl_xor_sync(0xffffffffu, v[0], o);
            v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
        }
    }
}

template <int NG>
__device__ __forceinline__ void scatter_to_red(const float (&v)[NG], float *red_q, int lane)
{
    if constexpr (NG >= 32) {
#pragma unroll
        for (int e = 0; e < NG / 32; ++e)
            red_q[lane * (NG / 32) + e] = v[e];
    } else {
        // each column's result sits on 32 / NG neighbouring lanes
        constexpr int rep = 32 / NG;
        if (lane % rep == 0)
            red_q[lane / rep] = v[0];
    }
}

// This thread's row of S^T (one token, NG query rows) in log2 units, with the
// tokens a row may not see set to -inf: past the chunk end, or past the row's
// causal limit L - (n_q - 1 - j) among the draft tokens.  The mask runs behind
// one branch that is taken only on a request's last tiles.  bf16 scores take the
// one factor scale * log2 e; E4M3 scores (hi plus lo part) the per-row factor at
// cf_addr (scale * log2 e * kv_scale * 2^e_row, the query row's power-of-two scale).
template <int NG, bool F8>
__device__ __forceinline__ void load_scores(uint32_t taddr, uint32_t lo_cols, float scale_log2,
                                            uint32_t cf_addr, bool tile_visible, int t, int t_end,
                                            int vis_all, int row0, int heads, float (&x)[NG])
{
    tmem_load_cols<NG>(taddr, x);
    if constexpr (F8) {
        // the lo part's scores sit lo_cols columns further on: the row's score is
        // the sum of the two (both in units of the query's 2^e)
        float y[NG];
        tmem_load_cols<NG>(taddr + lo_cols, y);
#pragma unroll
        for (int c = 0; c < NG; ++c)
            x[c] += y[c];
#pragma unroll
        for (int c4 = 0; c4 < NG; c4 += 4) {
            float f[4];
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3])
                         : "r"(cf_addr + 4 * c4));
#pragma unroll
            for (int e = 0; e < 4; ++e)
                x[c4 + e] *= f[e];
        }
    } else {
#pragma unroll
        for (int c = 0; c < NG; ++c)
            x[c] *= scale_log2;
    }
    if (!tile_visible) {
#pragma unroll
        for (int c = 0; c < NG; ++c) {
            const int lim = vis_all + (row0 + c) / heads;
            if (t >= lim || t >= t_end)
                x[c] = -INFINITY;
        }
    }
}

// Shift this thread's scores to x - m + p_off (m = the row's reference
// maximum; no shift while it is still -inf) and report whether any score lies
// more than tau above m.  A row whose m is -inf yields +inf for a visible score
// (flagged) and NaN for a masked one (ignored by fmaxf).
template <int NG, bool F8>
__device__ __forceinline__ bool shift_and_test(float (&x)[NG], uint32_t m_addr)
{
    using F = Fmt<F8>;
    float vmax = -INFINITY;
#pragma unroll
    for (int c4 = 0; c4 < NG; c4 += 4) {
        float m[4];
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(m[0]), "=f"(m[1]), "=f"(m[2]), "=f"(m[3])
                     : "r"(m_addr + 4 * c4));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            vmax = fmaxf(vmax, x[c4 + e] - m[e]);
            x[c4 + e] -= m[e] == -INFINITY ? 0.f : m[e] - F::p_off;
        }
    }
    return vmax > F::tau;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Q^T of one segment's query rows (row qrow on): bf16 nine 64-column blocks;
// E4M3 rows of 576 bytes: four latent blocks, then the 64-byte rope block
// through its own map, the hi part (rows of plane 0) and the lo part (plane 1,
// `planes` rows further on) of each.  Not inlined: it runs once per segment and
// keeps the kernel's code small.
template <int NG, bool F8>
__device__ __noinline__ void load_query(uint32_t s_q, const CUtensorMap *tm_qn,
                                        const CUtensorMap *tm_qr, int qrow, int planes,
                                        uint32_t bar_q)
{
    using L = Smem<NG, F8>;
    using F = Fmt<F8>;
    mbar_arrive_expect_tx(bar_q, L::q_bytes);
    if constexpr (F8) {
        const int qrow_lo = qrow + planes;
        for (int k = 0; k < F::sub - 1; ++k) {
            tma_load_2d(s_q + k * L::q_chunk, tm_qn, 128 * k, qrow, bar_q);
            tma_load_2d(s_q + k * L::q_chunk + L::q_lo, tm_qn, 128 * k, qrow_lo, bar_q);
        }
        tma_load_2d(s_q + (F::sub - 1) * L::q_chunk, tm_qr, kLatent, qrow, bar_q);
        tma_load_2d(s_q + (F::sub - 1) * L::q_chunk + L::q_rope_lo, tm_qr, kLatent, qrow_lo,
                    bar_q);
    } else {
        for (int k = 0; k < F::sub - 1; ++k)
            tma_load_2d(s_q + k * L::q_chunk, tm_qn, 64 * k, qrow, bar_q);
        tma_load_2d(s_q + (F::sub - 1) * L::q_chunk, tm_qr, 0, qrow, bar_q);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// The softmax warps' rare path: a score exceeds its reference maximum (always on
// a segment's first tile), or a wait gave up.  New reference maxima from the
// column maxima of x (which the reduction overwrites), the running sums and the
// O^T columns rescaled; a wait that gives up sets ok = false and leaves the
// enclosing loop.  One text for both score-load forms of the softmax below, so
// that each instantiation compiles the same statements.
#define PLMLA_SOFTMAX_RESCALE()                                                    \
    if (softmax_bar_or(!got || *abort_flag)) {                                     \
        ok = false;                                                                \
        break;                                                                     \
    }                                                                              \
    warp_reduce_scatter<CH, true>(x, lane);                                        \
    scatter_to_red<CH>(x, red + 64 * q + col0, lane);                              \
    softmax_bar();                                                                 \
    if (q == 0) {                                                                  \
        /* one warp per column half: new reference maxima and factors */           \
        bool any = false;                                                          \
        if (lane < CH) {                                                           \
            const int c = col0 + lane;                                             \
            const float mu = m_sm[c];                                              \
            /* the scores were shifted by mu (0 while unset): back to absolute */  \
            const float mx = fmaxf(fmaxf(red[c], red[64 + c]),                     \
                                   fmaxf(red[128 + c], red[192 + c])) +            \
                             (mu == -INFINITY ? 0.f : mu);                         \
            float alpha = 1.f;                                                     \
            if (mx != -INFINITY) {                                                 \
                if (mu == -INFINITY) {                                             \
                    m_sm[c] = mx;       /* first visible token of this row */      \
                    alpha = 0.f;                                                   \
                } else if (mx - mu > F::tau) {                                     \
                    m_sm[c] = mx;                                                  \
                    alpha = fast_exp2(mu - mx);                                    \
                }                                                                  \
            }                                                                      \
            al_sm[c] = alpha;                                                      \
            any = alpha != 1.f;                                                    \
        }                                                                          \
        any = __any_sync(0xffffffffu, any);                                        \
        if (lane == 0)                                                             \
            need_sm[h] = any ? 1 : 0;                                              \
    }                                                                              \
    softmax_bar();                                                                 \
    if (need_sm[h] != 0) {                                                         \
    _Pragma("unroll")                                                              \
        for (int c = 0; c < CH; ++c)                                               \
            lsum[c] *= ld_shared_f32(al_addr + 4 * c);                             \
    }                                                                              \
    if (i > 0 && (need_sm[0] | need_sm[1]) != 0) {                                 \
        /* O^T columns are rescaled once the previous P^T V is done */             \
        const bool done =                                                          \
            wait_bounded(bar_pv, (gt - 1) & 1, abort_flag, a.status, 8);           \
        if (softmax_bar_or(!done)) {                                               \
            ok = false;                                                            \
            break;                                                                 \
        }                                                                          \
        if (need_sm[h] != 0) {                                                     \
            tc_fence_after();                                                      \
    _Pragma("unroll")                                                              \
            for (int j = 0; j < 4; ++j)                                            \
                tmem_scale_cols<CH>(tmem + t_lane + 64 * j + col0, al_addr);       \
            tmem_wait_st();                                                        \
        }                                                                          \
    }

// V boxes of 2^b token rows (b < kTailMaps) for the rows of a request's last
// tile that lie inside its history.
constexpr int kTailMaps = 7;
struct TailMaps {
    CUtensorMap m[kTailMaps];
};

template <int NG, bool F8, int CL>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qr,
                 const __grid_constant__ TailMaps tail, const DecodeArgs a)
{
    using L = Smem<NG, F8>;
    using F = Fmt<F8>;
    static_assert(CL == 1 || (!F8 && (CL == 2 || CL == 4)), "cluster of teams: bf16 pages, 2 or 4");
    constexpr int NK = L::k_slots, NV = L::v_slots;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // The swizzled TMA boxes and MMA operands need 1024-byte alignment, and the
    // layout has no slack for it: with no static shared memory the dynamic base
    // is aligned.  Should it ever not be, report status 12 and touch nothing.
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the plan resets the status word
        if (threadIdx.x == 0)
            atomicExch(a.status, 12);
        return;
    }
    unsigned char *smem = smem_raw;
    const uint32_t s_k = smem_u32(smem);             // K ring
    const uint32_t s_v = s_k + L::v_off;             // V ring
    const uint32_t s_p = s_k + L::p_off;             // P^T
    const uint32_t s_q = s_k + L::q_off;             // Q^T
    const uint32_t bars = s_k + L::bar_off;
    const uint32_t bar_full_k = bars + kBarFullK;    // [NK] K item landed
    const uint32_t bar_empty_k = bars + kBarEmptyK;  // [NK] K slot free
    const uint32_t bar_full_v = bars + kBarFullV;    // [NV] V item ready
    const uint32_t bar_empty_v = bars + kBarEmptyV;  // [NV] V slot free
    const uint32_t bar_q = bars + kBarQ;             // Q^T landed
    const uint32_t bar_qe = bars + kBarQe;           // Q^T no longer read (segment's last S^T done)
    const uint32_t bar_s = bars + kBarS;             // [2] S^T of a tile complete, per buffer
    const uint32_t bar_sfree = bars + kBarSfree;     // [2] S^T buffer read by the softmax (128)
    const uint32_t bar_p = bars + kBarP;             // P^T of a tile written (128 arrivals)
    const uint32_t bar_pv = bars + kBarPv;           // P^T V of a tile complete
    const uint32_t bar_of = bars + kBarOf;           // O^T read out by the epilogue (128 arrivals)
    float *red = reinterpret_cast<float *>(smem + L::red_off);
    float *fin = reinterpret_cast<float *>(smem + L::fin_off);
    float *m_sm = reinterpret_cast<float *>(smem + L::m_off);
    float *al_sm = reinterpret_cast<float *>(smem + L::al_off);
    float *cf_sm = reinterpret_cast<float *>(smem + L::cf_off);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);
    volatile int *need_sm = reinterpret_cast<volatile int *>(smem + L::misc_off + 16);   // [2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_kv)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_qn)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_qr)) : "memory");
    }

    if (threadIdx.x == 0) {
        for (int k = 0; k < NK; ++k) {
            mbar_init(bar_full_k + 8 * k, 1);
            mbar_init(bar_empty_k + 8 * k, CL);        // a release from each CTA of the cluster
        }
        for (int k = 0; k < NV; ++k) {
            mbar_init(bar_full_v + 8 * k, 1);
            mbar_init(bar_empty_v + 8 * k, CL);
        }
        mbar_init(bar_q, 1);
        mbar_init(bar_qe, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_s + 8, 1);
        mbar_init(bar_sfree, kSoftmaxWarps);       // one arrival per softmax warp
        mbar_init(bar_sfree + 8, kSoftmaxWarps);
        mbar_init(bar_p, kSoftmaxWarps);
        mbar_init(bar_pv, 1);
        mbar_init(bar_of, kSoftmaxWarps);
        mbar_init(bars + kBarDrainS, 1);
        mbar_init(bars + kBarDrainPv, 1);
        for (int k = 0; k < 4; ++k)
            mbar_init(bars + kBarPvIssued + 8 * k, 1);
        *abort_flag = 0;
        need_sm[0] = 0;
        need_sm[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (warp == kWarpVProducer) {
        // V slots start at zero: a partial item leaves the rows past the history
        // untouched, and they must be finite (they meet zero probabilities)
        for (int off = 16 * lane; off < NV * F::v_slot; off += 16 * 32)
            st_shared_v4(s_v + off, 0u, 0u, 0u, 0u);
        fence_proxy_async();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // clustered teams: every CTA's barriers are initialised and its V slots
    // zeroed before any CTA multicasts into them
    if constexpr (CL > 1)
        cluster_sync();

    // everything above overlaps the plan kernel (programmatic dependent launch);
    // the schedule is read only once that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int cta = (int)blockIdx.x;
    // CL = 1: CTA = team * members + member.  CL > 1: the CTAs of a cluster are CL
    // teams of one member (they read the same KV items); cluster c holds teams
    // [(c % per) * CL, + CL) of member c / per, per = teams / CL.
    int team, member, rank = 0;
    if constexpr (CL == 1) {
        team = cta / a.members;
        member = cta % a.members;
    } else {
        rank = (int)cluster_rank();
        const int per = a.num_groups / CL;
        team = ((cta / CL) % per) * CL + rank;
        member = (cta / CL) / per;
    }
    const int row0 = team * NG;
    const int seg_begin = a.seg_member_indptr[member];
    const int seg_end = a.seg_member_indptr[member + 1];   // empty range: no work
    const int seg_total = *a.seg_count;
    // the combine kernel may launch now: it occupies SMs only as CTAs of this
    // grid exit, and waits per request on the finished-segment counters
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ---------------------------------------------------------- K producer
        if (lane == 0) {
            // the latent blocks are read again (as V items) shortly: keep them in
            // L2 until then; the rope block is not
            const uint64_t pol_keep = l2_policy_evict_last();
            const uint64_t pol_once = l2_policy_evict_first();
            int slot = 0;
            uint32_t phase = 0;
            int issued = 0;                          // K items issued (all segments)
            int q_loads = 0;
            bool ok = true;
            // Q^T of segment s: the buffer is free once the previous segment's last
            // S^T has completed (bar_qe)
            auto load_q = [&](int s) -> bool {
                const int local = s - seg_begin;
                if (local > 0 && !wait_bounded(bar_qe, (local - 1) & 1, abort_flag, a.status, 1))
                    return false;
                const int qrow = a.segments[s].x * a.rows_per_req + row0;
                load_query<NG, F8>(s_q, &tm_qn, &tm_qr, qrow, a.num_reqs * a.rows_per_req, bar_q);
                ++q_loads;
                return true;
            };
            if constexpr (F8) {
                // E4M3 pages: each segment's Q^T before its K items (measured faster
                // for this variant than the deferred order below)
                for (int s = seg_begin; s < seg_end && ok; ++s) {
                    const int4 seg = a.segments[s];
                    if (!load_q(s)) {
                        ok = false;
                        break;
                    }
                    const int32_t *trow = a.page_table + (int64_t)seg.x * a.table_ld;
                    const int n_tiles = (seg.z - seg.y + kTile - 1) / kTile;
                    for (int i = 0; i < n_tiles && ok; ++i) {
                        const int t = seg.y + i * kTile;
                        const int page = trow[t / kPageTokens];
                        const int tok = t % kPageTokens;
                        // the producers' and issuers' item loops stay rolled: the kernel is
                        // bound by instruction fetch as much as by its streams
#pragma unroll 1
                        for (int k = 0; k < F::sub; ++k) {
                            if (!wait_bounded(bar_empty_k + 8 * slot, phase ^ 1, abort_flag,
                                              a.status, 2)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(bar_full_k + 8 * slot, kSubBytes);
                            tma_load_3d_hint(s_k + slot * kSubBytes, &tm_kv, F::col_step * k, tok,
                                             page, bar_full_k + 8 * slot,
                                             k < F::sub - 1 ? pol_keep : pol_once);
                            ++issued;
                            if (++slot == NK) {
                                slot = 0;
                                phase ^= 1;
                            }
                        }
                    }
                }
            } else {
                // A segment's first K items go out before its Q^T: their ring slots are
                // freed by S^T of the previous segment's items, which needs no new Q^T,
                // so the HBM stream keeps going while that S^T finishes.  Q^T of the
                // `pending` segment must be loaded before K item `q_deadline` (the first
                // item whose slot only this segment's S^T can free).
                int pending = -1, q_deadline = 0;
                for (int s = seg_begin; s < seg_end && ok; ++s) {
                    const int local = s - seg_begin;
                    const int4 seg = a.segments[s];
                    if (pending >= 0) {                  // a segment of fewer than NK items
                        if (!load_q(pending)) {
                            ok = false;
                            break;
                        }
                        pending = -1;
                    }
                    if (local == 0) {
                        if (!load_q(s)) {
                            ok = false;
                            break;
                        }
                    } else {
                        pending = s;
                        q_deadline = issued + NK;
                    }
                    const int32_t *trow = a.page_table + (int64_t)seg.x * a.table_ld;
                    const int n_tiles = (seg.z - seg.y + kTile - 1) / kTile;
                    for (int i = 0; i < n_tiles && ok; ++i) {
                        const int t = seg.y + i * kTile;
                        const int page = trow[t / kPageTokens];
                        const int tok = t % kPageTokens;
                        // Entering a page: warm the address translations of the next page
                        // this CTA reads (the segment's next page, else the next segment's
                        // first) with one-row L2 prefetches of its first row and of the
                        // first row past a 2 MiB boundary inside it, a page's worth of
                        // tiles before the ring reaches it.  Measured: ~2% off the steady
                        // step.
                        if (i == 0 || tok == 0) {
                            const int tn = (t / kPageTokens + 1) * kPageTokens;
                            int np = -1, nt0 = 0;
                            if (tn < seg.z) {
                                np = trow[tn / kPageTokens];
                            } else if (s + 1 < seg_end) {
                                const int4 nx = a.segments[s + 1];
                                np = a.page_table[(int64_t)nx.x * a.table_ld + nx.y / kPageTokens];
                                nt0 = nx.y % kPageTokens;
                            }
                            if (np >= 0) {
                                tma_prefetch_3d(&tail.m[0], 0, nt0, np);
                                const uint64_t pa = reinterpret_cast<uint64_t>(a.slab) +
                                                    (uint64_t)np * (uint64_t)a.page_stride * 2u;
                                const uint64_t nb = ((pa >> 21) + 1) << 21;
                                const uint64_t rb = (uint64_t)kRow * 2u;
                                const int tb = (int)((nb - pa + rb - 1) / rb);
                                if (tb > nt0 && tb < kPageTokens)
                                    tma_prefetch_3d(&tail.m[0], 0, tb, np);
                            }
                        }
#pragma unroll 1
                        for (int k = 0; k < F::sub; ++k) {
                            if (pending >= 0 && issued >= q_deadline) {
                                if (!load_q(pending)) {
                                    ok = false;
                                    break;
                                }
                                pending = -1;
                            }
                            if (!wait_bounded(bar_empty_k + 8 * slot, phase ^ 1, abort_flag,
                                              a.status, 2)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(bar_full_k + 8 * slot, kSubBytes);
                            // clustered teams take turns: item n comes from CTA n % CL
                            if (CL == 1 || issued % CL == rank)
                                kv_load<CL>(s_k + slot * kSubBytes, &tm_kv, F::col_step * k, tok,
                                            page, bar_full_k + 8 * slot,
                                            k < F::sub - 1 ? pol_keep : pol_once);
                            ++issued;
                            if (++slot == NK) {
                                slot = 0;
                                phase ^= 1;
                            }
                        }
                    }
                }
                // the last segment's Q^T, if it still waits (fewer than NK items)
                if (ok && pending >= 0)
                    load_q(pending);
            }
            // every issued copy must land before the CTA can exit: the last NK
            // items may still be in flight, earlier ones were consumed
            if (q_loads > 0)
                wait_drain(bar_q, (q_loads - 1) & 1);
            for (int it = issued > NK ? issued - NK : 0; it < issued; ++it)
                wait_drain(bar_full_k + 8 * (it % NK), (uint32_t)(it / NK) & 1u);
        }
    } else if (warp == kWarpVProducer) {
        // ---------------------------------------------------------- V producer
        // V item v of a tile = latent block v / v_per_block (128 latent columns: two
        // 64-column boxes for bf16, one 128-byte box for E4M3), the tile's tokens
        // [(v % v_per_block) * v_tokens, + v_tokens).
        // In a request's last tile an item loads only its rows inside the history,
        // as boxes of power-of-two heights (the tail maps) issued together; the
        // rows past the history keep what the slot held before -- zeros written
        // at the start of the kernel or history rows of an earlier item, finite
        // either way -- and their probabilities are zero.  An item wholly past the
        // history loads nothing and is released at once.
        const uint64_t pol_once = l2_policy_evict_first();   // the tile's last read
        int slot = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int s = seg_begin; s < seg_end && ok; ++s) {
            const int4 seg = a.segments[s];
            const int32_t *trow = a.page_table + (int64_t)seg.x * a.table_ld;
            const int n_tiles = (seg.z - seg.y + kTile - 1) / kTile;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int t = seg.y + i * kTile;
                const int page = trow[t / kPageTokens];
                const int tok = t % kPageTokens;
#pragma unroll 1
                for (int v = 0; v < F::v_items; ++v) {
                    // first token of the item within the tile
                    const int toff = (v % F::v_per_block) * F::v_tokens;
                    bool got = true;
                    if (lane == 0)
                        got = wait_bounded(bar_empty_v + 8 * slot, phase ^ 1, abort_flag, a.status,
                                           11);
                    if (lane == 0 && got) {
                        // clustered teams take turns: item n comes from CTA n % CL (the
                        // others only expect its bytes)
                        const bool mine = CL == 1 || issued % CL == rank;
                        const uint32_t dst = s_v + slot * F::v_slot;
                        const uint32_t fb = bar_full_v + 8 * slot;
                        const int col = 128 * (v / F::v_per_block), tk = tok + toff;
                        // rows of the item inside the history
                        const int live = seg.z - (t + toff);
                        if (live >= F::v_tokens) {
                            mbar_arrive_expect_tx(fb, F::v_slot);
                            if (mine) {
                                kv_load<CL>(dst, &tm_v, col, tk, page, fb, pol_once);
                                if constexpr (!F8)
                                    kv_load<CL>(dst + kVHalf, &tm_v, col + 64, tk, page, fb,
                                                pol_once);
                            }
                        } else if (live <= 0) {
                            mbar_arrive(fb);
                        } else {
                            constexpr int halves = F8 ? 1 : 2;
                            mbar_arrive_expect_tx(fb, (uint32_t)(live * 128 * halves));
                            int r0 = 0;
#pragma unroll 1
                            for (int b = kTailMaps - 1; b >= 0 && mine; --b) {
                                if ((live >> b) & 1) {
                                    kv_load<CL>(dst + r0 * 128, &tail.m[b], col, tk + r0, page, fb,
                                                pol_once);
                                    if constexpr (!F8)
                                        kv_load<CL>(dst + kVHalf + r0 * 128, &tail.m[b], col + 64,
                                                    tk + r0, page, fb, pol_once);
                                    r0 += 1 << b;
                                }
                            }
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
                        ok = false;
                        break;
                    }
                    ++issued;
                    if (++slot == NV) {
                        slot = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (lane == 0) {
            // copies still in flight: at most the last NV items
            for (int back = 0; back < NV && back < issued; ++back) {
                const int it = issued - 1 - back;
                wait_drain(bar_full_v + 8 * (it % NV), (uint32_t)(it / NV) & 1u);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- S^T issuer
        if (lane == 0) {
            bool issued = false, ok = true;
            constexpr uint32_t idesc_s = idesc_for<F8>(128, F::s_rows * NG, false, false);
            const uint64_t dk0 = sdesc(s_k, 16, 1024, kSw128);
            const uint64_t dq0 = sdesc(s_q, 16, 1024, kSw128);
            const uint64_t dq_rope =
                sdesc(s_q + (F::sub - 1) * L::q_chunk, 16, F8 ? 512 : 1024, F8 ? kSw64 : kSw128);
            int slot = 0;
            uint32_t phase = 0;
            int g = 0;                               // tiles so far (all segments)
            for (int s = seg_begin; s < seg_end && ok; ++s) {
                const int local = s - seg_begin;
                const int4 seg = a.segments[s];
                const int n_tiles = (seg.z - seg.y + kTile - 1) / kTile;
                if (!wait_bounded(bar_q, local & 1, abort_flag, a.status, 3)) {
                    ok = false;
                    break;
                }
                for (int i = 0; i < n_tiles; ++i, ++g) {
                    const uint32_t b = g & 1;
                    // the softmax of tile g - 2 must be done with this S^T buffer, and
                    // S^T runs at most kLead<F8> tiles ahead of P^T V, so that a tile's
                    // latent blocks are still in L2 when they are read again as V items
                    if (g >= 2 && !wait_bounded(bar_sfree + 8 * b, ((g - 2) >> 1) & 1, abort_flag,
                                                a.status, 13)) {
                        ok = false;
                        break;
                    }
                    constexpr int lead = kLead<F8>;
                    static_assert(lead >= 1 && lead <= 3, "lead");
                    if (g >= lead &&
                        !wait_bounded(bars + kBarPvIssued + 8 * ((g - lead) & 3),
                                      ((g - lead) >> 2) & 1, abort_flag, a.status, 10)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_s = tmem + kTmemS + F::s_stride * b;
                    // not unrolled: the issuers' code competes with the softmax warps'
                    // for the instruction cache (measured: steady decode -4%, E4M3 -11%)
#pragma unroll 1
                    for (int k = 0; k < F::sub; ++k) {
                        if (!wait_bounded(bar_full_k + 8 * slot, phase, abort_flag, a.status, 4)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t da = dk0 + (uint64_t)(slot * (kSubBytes >> 4));
                        // 32-byte K steps inside the 128-byte swizzled rows
                        constexpr int last_mmas = F::rope_mmas;
                        const int n_mma = k == F::sub - 1 ? last_mmas : 4;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            if (kk < n_mma) {
                                // the E4M3 rope block of Q^T has 64-byte rows
                                const uint64_t db =
                                    (F8 && k == F::sub - 1) ? dq_rope + 2 * kk
                                                            : dq0 + (uint64_t)(k * (L::q_chunk >> 4) + 2 * kk);
                                mma<F8>(d_s, da + 2 * kk, db, idesc_s, (k | kk) != 0);
                            }
                        mma_commit_all<CL>(bar_empty_k + 8 * slot);
                        issued = true;
                        if (++slot == NK) {
                            slot = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok)
                        break;
                    mma_commit(bar_s + 8 * b);
                    if (i == n_tiles - 1)
                        mma_commit(bar_qe);
                }
            }
            if (issued) {
                mma_commit(bars + kBarDrainS);
                wait_drain(bars + kBarDrainS, 0);
            }
        }
    } else if (warp == kWarpPvIssuer) {
        // ----------------------------------------------------- P^T V issuer
        if (lane == 0) {
            bool issued = false, ok = true;
            constexpr uint32_t idesc_pv = idesc_for<F8>(128, L::pn, true, true);
            constexpr uint32_t p_layout = layout_for_row(L::p_row);
            // MN-major operands: 8-token row groups 1024 bytes (V) and 8 P^T rows apart
            const uint64_t dv0 = sdesc(s_v, kVHalf, 1024, kSw128);
            const uint64_t dp0 = sdesc(s_p, 8192, 8 * L::p_row, p_layout);
            int slot = 0;
            uint32_t phase = 0;
            int g = 0;
            for (int s = seg_begin; s < seg_end && ok; ++s) {
                const int local = s - seg_begin;
                const int4 seg = a.segments[s];
                const int n_tiles = (seg.z - seg.y + kTile - 1) / kTile;
                for (int i = 0; i < n_tiles; ++i, ++g) {
                    // O^T of the previous segment must have been read out
                    if (i == 0 && local > 0 &&
                        !wait_bounded(bar_of, (local - 1) & 1, abort_flag, a.status, 5)) {
                        ok = false;
                        break;
                    }
                    if (!wait_bounded(bar_p, g & 1, abort_flag, a.status, 6)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // not unrolled either, except in the clustered variant, whose extend
                    // workload lost 3% to it (the single-team and E4M3 variants gained a
                    // further 0-6%)
#pragma unroll(CL == 1 ? 1 : F::v_items)
                    for (int v = 0; v < F::v_items; ++v) {
                        if (!wait_bounded(bar_full_v + 8 * slot, phase, abort_flag, a.status, 14)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t da = dv0 + (uint64_t)(slot * (F::v_slot >> 4));
                        // O^T block j; the item's first token h within the tile
                        const int j = v / F::v_per_block, h = (v % F::v_per_block) * F::v_tokens;
                        // each MMA takes 16 (bf16) or 32 (E4M3) tokens: 2 or 4 row groups
                        constexpr int k_tok = F8 ? 32 : 16;
#pragma unroll
                        for (int kk = 0; kk < F::v_tokens / k_tok; ++kk)
                            mma<F8>(tmem + 64 * j, da + (uint64_t)((k_tok * 128 >> 4) * kk),
                                    dp0 + (uint64_t)(((h + k_tok * kk) * L::p_row) >> 4),
                                    idesc_pv, (i | h | kk) != 0);
                        mma_commit_all<CL>(bar_empty_v + 8 * slot);
                        issued = true;
                        if (++slot == NV) {
                            slot = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok)
                        break;
                    mma_commit(bar_pv);
                    mbar_arrive(bars + kBarPvIssued + 8 * (g & 3));
                }
            }
            if (issued) {
                mma_commit(bars + kBarDrainPv);
                wait_drain(bars + kBarDrainPv, 0);
            }
        }
    } else {
        // ------------------------------------------------------------- softmax
        // warp w in 2..9: TMEM lane quadrant w % 4 (tokens of S^T, latent rows of
        // O^T), columns [h*CH, (h+1)*CH) of the NG query rows, h = (w - 2) / 4
        constexpr int CH = NG / 2;
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int col0 = h * CH;
        const int tok = 32 * q + lane;          // token lane of S^T / latent row of O^T
        const int st = threadIdx.x - 64;        // 0..255
        const uint32_t t_lane = (uint32_t)(32 * q) << 16;
        const uint32_t m_addr = smem_u32(m_sm) + 4 * col0;
        const uint32_t al_addr = smem_u32(al_sm) + 4 * col0;
        const uint32_t cf_addr = smem_u32(cf_sm) + 4 * col0;
        // E4M3 with fewer than 32 query rows: the P^T rows are padded to 32 bytes
        // and the padding stays zero (the P^T V MMA multiplies it into unused columns)
        if constexpr (L::pn > NG) {
            for (int r = st; r < kTile; r += kSoftmaxThreads) {
                const uint32_t off = (uint32_t)(r * L::p_row + 16);
                st_shared_v4(s_p + (off ^ (((off >> 7) & 1u) << 4)), 0u, 0u, 0u, 0u);
            }
        }
        bool ok = true;
        int gt = 0;
        for (int s = seg_begin; s < seg_end && ok; ++s) {
            const int local = s - seg_begin;
            const int4 seg = a.segments[s];
            const int n_tiles = (seg.z - seg.y + kTile - 1) / kTile;
            const int Lr = a.seq_lens[seg.x];
            const int vis_all = Lr - (a.n_q - 1);   // tokens below this are visible to every row
            if (local > 0)
                softmax_bar();                       // previous epilogue is done with m_sm
            for (int c = st; c < NG; c += kSoftmaxThreads) {
                m_sm[c] = -INFINITY;
                if constexpr (F8) {
                    // score factor of query row c: scale * log2 e * kv_scale * 2^e
                    const int e = a.qexp[(int64_t)seg.x * a.rows_per_req + row0 + c];
                    cf_sm[c] = a.scale_log2 * a.kv_scale * __uint_as_float((uint32_t)(e + 127) << 23);
                }
            }
            softmax_bar();
            float lsum[CH];
#pragma unroll
            for (int c = 0; c < CH; ++c)
                lsum[c] = 0.f;

            for (int i = 0; i < n_tiles; ++i, ++gt) {
                const int t_base = seg.y + i * kTile;
                const int t = t_base + tok;
                const bool tile_visible = t_base + kTile <= vis_all;
                const uint32_t b = gt & 1;
                const uint32_t s_col = kTmemS + F::s_stride * b + col0;
                // warp-uniform, because tcgen05.ld below is a .sync.aligned instruction
                const bool got = __all_sync(
                    0xffffffffu, wait_bounded(bar_s + 8 * b, (gt >> 1) & 1, abort_flag, a.status, 7));
                float x[CH];
                if constexpr (CL == 1) {
                    bool exceed = false;
                    if (got) {
                        tc_fence_after();
                        load_scores<CH, F8>(tmem + t_lane + s_col, NG, a.scale_log2, cf_addr,
                                            tile_visible, t, seg.z, vis_all, row0 + col0,
                                            a.num_heads, x);
                        exceed = shift_and_test<CH, F8>(x, m_addr);
                    }
                    if (softmax_bar_or(exceed || !got || *abort_flag)) {
                        PLMLA_SOFTMAX_RESCALE();
                        load_scores<CH, F8>(tmem + t_lane + s_col, NG, a.scale_log2, cf_addr,
                                            tile_visible, t, seg.z, vis_all, row0 + col0,
                                            a.num_heads, x);
                        shift_and_test<CH, F8>(x, m_addr);
                    }
                } else {
                    // clustered teams: one copy of the score load, taken again after a
                    // rescale (measured 5% faster for this variant on the 4-draft decode,
                    // 3% slower for the single-team one)
                    bool rescaled = false;
#pragma unroll 1
                    for (;;) {
                        bool exceed = false;
                        if (got) {
                            tc_fence_after();
                            load_scores<CH, F8>(tmem + t_lane + s_col, NG, a.scale_log2, cf_addr,
                                                tile_visible, t, seg.z, vis_all, row0 + col0,
                                                a.num_heads, x);
                            exceed = shift_and_test<CH, F8>(x, m_addr);
                        }
                        if (rescaled || !softmax_bar_or(exceed || !got || *abort_flag))
                            break;
                        PLMLA_SOFTMAX_RESCALE();
                        rescaled = true;
                    }
                    if (!ok)
                        break;
                }
                // this S^T buffer may now be overwritten by the tile after next
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_sfree + 8 * b);
                // probabilities 2^(x - m + p_off) (x is already shifted) and running
                // sums (of the fp32 values; only the MMA operand is rounded)
                constexpr int kWords = F8 ? CH / 4 : CH / 2;
                uint32_t pk[kWords];
                if constexpr (F8) {
#pragma unroll
                    for (int c = 0; c < CH; c += 4) {
                        float p[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            p[e] = fast_exp2(x[c + e]);       // 2^-inf = 0
                            lsum[c + e] += p[e];
                        }
                        pk[c / 4] = (uint32_t)e4m3x2(p[0], p[1]) | ((uint32_t)e4m3x2(p[2], p[3]) << 16);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < CH; c += 2) {
                        const float p0 = fast_exp2(x[c]);    // 2^-inf = 0
                        const float p1 = fast_exp2(x[c + 1]);
                        lsum[c] += p0;
                        lsum[c + 1] += p1;
                        pk[c / 2] = pack_bf16x2(p0, p1);
                    }
                }
                // P^T is free once the previous tile's P^T V has completed
                if (gt > 0) {
                    const bool done =
                        wait_bounded(bar_pv, (gt - 1) & 1, abort_flag, a.status, 8);
                    if (softmax_bar_or(!done)) {
                        ok = false;
                        break;
                    }
                }
                {
                    // this token's row of P^T (p_row bytes, 16-byte chunks swizzled
                    // like the MMA operand); this thread writes its column half
                    constexpr int row_bytes = L::p_row;
                    constexpr int swz_bits = row_bytes == 128 ? 3 : (row_bytes == 64 ? 2 : 1);
                    constexpr int my_bytes = kWords * 4;
                    if constexpr (my_bytes >= 16) {
#pragma unroll
                        for (int ch = 0; ch < my_bytes / 16; ++ch) {
                            const uint32_t off =
                                (uint32_t)(tok * row_bytes + h * my_bytes + 16 * ch);
                            const uint32_t sw = off ^ (((off >> 7) & ((1u << swz_bits) - 1u)) << 4);
                            st_shared_v4(s_p + sw, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2],
                                         pk[4 * ch + 3]);
                        }
                    } else {
                        // 8 bytes (E4M3, 16 query rows): half of a 16-byte chunk
                        const uint32_t off = (uint32_t)(tok * row_bytes + h * my_bytes);
                        const uint32_t sw = off ^ (((off >> 7) & ((1u << swz_bits) - 1u)) << 4);
                        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(s_p + sw),
                                     "r"(pk[0]), "r"(pk[1])
                                     : "memory");
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_p);
            }
            if (!ok)
                break;

            // ---- segment epilogue: normalised partial state of the segment
            const bool done = wait_bounded(bar_pv, (gt - 1) & 1, abort_flag, a.status, 9);
            if (softmax_bar_or(!done)) {
                ok = false;
                break;
            }
            tc_fence_after();
            warp_reduce_scatter<CH, false>(lsum, lane);
            scatter_to_red<CH>(lsum, red + 64 * q + col0, lane);
            softmax_bar();
            if (q == 0 && lane < CH) {
                const int c = col0 + lane;
                const float l = red[c] + red[64 + c] + red[128 + c] + red[192 + c];
                // 1 / row sum (0 for an empty row); E4M3 values carry kv_scale
                fin[c] = l > 0.f ? (F8 ? a.kv_scale : 1.f) / l : 0.f;
                a.lse_part[(int64_t)(team * seg_total + s) * NG + c] =
                    l > 0.f ? (m_sm[c] + log2f(l) - F::p_off) * kLn2 : -INFINITY;
            }
            softmax_bar();
            // normalised partial output: thread = latent row of each O^T block;
            // for a fixed row the 128 threads of a column half store 512
            // contiguous bytes
            const uint32_t inv_addr = smem_u32(fin) + 4 * col0;
            float *out0 = a.o_part + ((int64_t)(team * seg_total + s) * NG + col0) * kLatent + tok;
            float inv[CH];
#pragma unroll
            for (int c = 0; c < CH; ++c)
                inv[c] = ld_shared_f32(inv_addr + 4 * c);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float o[CH];
                tmem_load_cols<CH>(tmem + t_lane + 64 * j + col0, o);
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    out0[(int64_t)c * kLatent + 128 * j] = o[c] * inv[c];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_of);
            // publish the segment: every thread's stores, then one counter update
            __threadfence();
            softmax_bar();
            if (st == 0)
                atomicAdd(a.done + team * a.num_reqs + seg.x, 1);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
    }
    // clustered teams: no CTA leaves while another may still write into its
    // shared memory or arrive on its barriers (every wait above is bounded, so
    // every thread of the cluster gets here)
    if constexpr (CL > 1)
        cluster_sync();
}

#undef PLMLA_SOFTMAX_RESCALE

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, int rank,
              const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    // out-of-range elements (the E4M3 rope block's columns past 576) read as zero
    return fn(map, dtype, rank, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps over the slab (K items, V items, and the V tail boxes), kept for
// the last slab seen by this host thread: they depend only on the slab's
// address, page count, page stride and format.
struct KvMaps {
    CUtensorMap kv, v;
    TailMaps tail;
};

bool kv_maps(const DecodeArgs &a, bool f8, KvMaps *out)
{
    thread_local struct {
        bool valid;
        const void *slab;
        int64_t pages, stride;
        bool f8;
        KvMaps maps;
    } cache = {};
    if (cache.valid && cache.slab == a.slab && cache.pages == a.num_pages &&
        cache.stride == a.page_stride && cache.f8 == f8) {
        *out = cache.maps;
        return true;
    }
    const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t esize = f8 ? 1 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)kRow, (cuuint64_t)kPageTokens, (cuuint64_t)a.num_pages};
    const cuuint64_t strides[2] = {(cuuint64_t)kRow * esize, (cuuint64_t)a.page_stride * esize};
    // one box row is 128 bytes: 64 bf16 or 128 E4M3 columns
    const cuuint32_t cols = f8 ? 128 : 64;
    const cuuint32_t kv_box[3] = {cols, (cuuint32_t)kTile, 1};
    const cuuint32_t v_box[3] = {cols, (cuuint32_t)(f8 ? Fmt<true>::v_tokens : Fmt<false>::v_tokens),
                                 1};
    KvMaps m;
    if (!make_map(&m.kv, dt, a.slab, 3, dims, strides, kv_box) ||
        !make_map(&m.v, dt, a.slab, 3, dims, strides, v_box))
        return false;
    for (int b = 0; b < kTailMaps; ++b) {
        const cuuint32_t rows = 1u << b;
        const cuuint32_t box[3] = {cols, rows < v_box[1] ? rows : v_box[1], 1};
        if (!make_map(&m.tail.m[b], dt, a.slab, 3, dims, strides, box))
            return false;
    }
    cache.valid = true;
    cache.slab = a.slab;
    cache.pages = a.num_pages;
    cache.stride = a.page_stride;
    cache.f8 = f8;
    cache.maps = m;
    *out = m;
    return true;
}

// Query maps: bf16 q_nope (64-column boxes) and q_rope, or the two-part E4M3
// rows [2 * R*n_q*H, 576] (hi plane, then lo plane): 128-byte boxes for the
// latent, a 64-byte box (64-byte swizzle) for the rope.
template <int NG>
bool q_maps(const DecodeArgs &a, bool f8, CUtensorMap *qn, CUtensorMap *qr)
{
    const cuuint64_t rows = (cuuint64_t)a.num_reqs * a.rows_per_req;
    if (f8) {
        const cuuint64_t q_dims[2] = {(cuuint64_t)kRow, 2 * rows};
        const cuuint64_t q_strides[1] = {(cuuint64_t)kRow};
        const cuuint32_t q_box[2] = {128, (cuuint32_t)NG};
        const cuuint32_t r_box[2] = {64, (cuuint32_t)NG};
        return make_map(qn, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q8, 2, q_dims, q_strides, q_box) &&
               make_map(qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q8, 2, q_dims, q_strides, r_box,
                        CU_TENSOR_MAP_SWIZZLE_64B);
    }
    const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t qn_dims[2] = {(cuuint64_t)kLatent, rows};
    const cuuint64_t qn_strides[1] = {(cuuint64_t)kLatent * 2};
    const cuuint64_t qr_dims[2] = {(cuuint64_t)kRope, rows};
    const cuuint64_t qr_strides[1] = {(cuuint64_t)kRope * 2};
    const cuuint32_t q_box[2] = {64, (cuuint32_t)NG};
    return make_map(qn, bf16, a.q_nope, 2, qn_dims, qn_strides, q_box) &&
           make_map(qr, bf16, a.q_rope, 2, qr_dims, qr_strides, q_box);
}

template <int NG, bool F8, int CL>
cudaError_t launch_ng(const DecodeArgs &a, cudaStream_t stream)
{
    KvMaps kv;
    CUtensorMap qn, qr;
    if (!kv_maps(a, F8, &kv) || !q_maps<NG>(a, F8, &qn, &qr))
        return cudaErrorInvalidValue;
    constexpr int smem = Smem<NG, F8>::alloc;
    cudaError_t err = cudaFuncSetAttribute(decode_tc_kernel<NG, F8, CL>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.members * (unsigned)a.num_groups);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<NG, F8, CL>, kv.kv, kv.v, qn, qr, kv.tail, a);
}

// Clusters of CL decode CTAs (64-row teams, bf16 pages) that the device holds at
// once, or 0.
template <int CL>
int max_clusters_of()
{
    constexpr int smem = Smem<64, false>::alloc;
    if (cudaFuncSetAttribute(decode_tc_kernel<64, false, CL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<64, false, CL>, &cfg) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

int decode_cluster_teams(int group_rows, int groups, bool fp8, int max_teams)
{
    if (fp8 || group_rows != 64)
        return 1;
    if (max_teams >= 4 && groups % 4 == 0)
        return 4;
    return max_teams >= 2 && groups % 2 == 0 ? 2 : 1;
}

int decode_max_clusters(int cluster)
{
    static int cached[64][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 0;
    const int k = cluster == 4 ? 1 : 0;
    if (cluster != 2 && cluster != 4)
        return 0;
    if (dev < 64 && cached[dev][k] > 0)
        return cached[dev][k];
    const int n = cluster == 4 ? max_clusters_of<4>() : max_clusters_of<2>();
    if (dev < 64 && n > 0)
        cached[dev][k] = n;
    return n;
}

cudaError_t launch_decode_tc(const DecodeArgs &args, cudaStream_t stream)
{
    if (args.fp8) {
        switch (args.group_rows) {
        case 64: return launch_ng<64, true, 1>(args, stream);
        case 32: return launch_ng<32, true, 1>(args, stream);
        case 16: return launch_ng<16, true, 1>(args, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (args.group_rows) {
    case 64:
        if (args.cluster == 4)
            return launch_ng<64, false, 4>(args, stream);
        if (args.cluster == 2)
            return launch_ng<64, false, 2>(args, stream);
        return launch_ng<64, false, 1>(args, stream);
    case 32: return launch_ng<32, false, 1>(args, stream);
    case 16: return launch_ng<16, false, 1>(args, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace plmla
