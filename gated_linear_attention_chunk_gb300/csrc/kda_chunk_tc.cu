// Chunked (64-token) KDA forward on tcgen05 tensor cores, bf16 inputs, dk = dv = 128.
//
// The recurrence is the gated delta rule with per-channel decay ("Kimi K3 on
// Fireworks: Fast RL at frontier scale", KDA paragraph: chunk-parallel training
// of linear attention whose compact recurrent state is updated with
// channel-wise gating; the kernel fuses the chunk-local work and keeps the
// state on chip so intermediates never touch HBM).  Unrolled over one chunk of
// C = 64 tokens with state S (dk x dv) at the chunk start, alpha_r = exp(g_r),
// A_r = prod_{j<=r} alpha_j (prefix products, per channel), A_C = A_63:
//
//   Kbar = K * A,  Qbar = scale * Q * A,  Ktil = K / A          (row-wise, per channel)
//   M[r,i] = beta_r Kbar_r . Ktil_i  (i < r),   P[r,i] = Qbar_r . Ktil_i  (i <= r)
//   T' = (I + M)^-1 Diag(beta),  W = T' Kbar,  Utl = T' V
//   U = Utl - W S,   O = Qbar S + P U,   S <- Diag(A_C) (S + Ktil^T U)
//
// Every factor stays bounded except Ktil (<= 1/A_C); the kernel therefore
// requires A_C >= 2^-100 per channel and chunk (checked: such a chain is flagged
// for the token-sequential kernel, or KDA_ERR_GATE_RANGE without room for the flag).
//
// One CTA per (sequence, head) walks its full chunks in order.  Warp roles:
//   warp 0       TMA producer: q, k, g, v tiles (SW128) + beta, 2-stage ring
//   warp 1       chain MMA issuer (and TMEM owner)
//   warp 2       prep MMA issuer (polls both prep products)
//   warps 4-7    chain group: W tile from W^T, U and state epilogues in TMEM, O to HBM
//   warps 8-15   decay group: prefix products, Kbar / Qbar / Ktil in place
//   warps 16-19  solve group: M and P from the accumulator, T' = (I+M)^-1 Diag(beta)
// Registers are split per warpgroup with setmaxnreg (the control warps need few).
// The decay group runs up to one chunk ahead of the solve group, which runs one
// chunk ahead of the chain.  The state lives in TMEM transposed (lane = value
// column j, column = channel c) as an fp32 master plus a bf16 copy that feeds
// the next chunk's MMAs as the A operand straight from TMEM.
//
// Every mbarrier wait is bounded (about one second); a wait that gives up sets
// the timeout bit in the status word, and all roles drain and exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "kda_internal.h"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk length
constexpr int kD = 128;         // dk = dv
constexpr int kThreads = 640;   // 20 warps
constexpr uint64_t kWaitNs = 1000000000ull;

// dynamic shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kStage = 65536;                 // per-stage: R (k|q, 32K), G (16K), V (16K)
constexpr uint32_t OFF_R = 0, OFF_G = 32768, OFF_V = 49152;
// The W tile of a chunk (MN-major, row = channel) is written over the Kbar half of
// its R tile once Kbar's last reader (the W / Utl product) has completed.
constexpr uint32_t OFF_P = 2 * kStage;             // 2 x 8K    P (K-major: row = token)
constexpr uint32_t OFF_TT = OFF_P + 2 * 8192;      // 2 x 8K    T' (K-major), by chunk parity
constexpr int kLdM = 68;                           // row stride (floats) of the fp32 M buffer (16-byte rows)
constexpr int kLdT = 72;                           // row stride of the fp32 T buffer (16-byte rows)
constexpr int kLdX = 40;                           // row stride of the block-product scratch
constexpr uint32_t OFF_M = OFF_TT + 2 * 8192;      // fp32 64 x kLdM
constexpr uint32_t OFF_T = OFF_M + 64 * kLdM * 4;  // fp32 64 x kLdT
constexpr uint32_t kDynSmem = OFF_T + 64 * kLdT * 4 + 1024;

// TMEM columns (512 allocated)
constexpr uint32_t TM_S = 0, TM_SB = 128, TM_U = 192, TM_W = 256, TM_UB = 320, TM_O = 352, TM_PREP = 416;

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_g, tm_v;
    const __nv_bfloat16 *beta;
    __nv_bfloat16 *o;
    const int32_t *order;         // launch order of the sequences, or null
    const int32_t *cu;
    const float *init_state;
    float *state_out;
    uint32_t *status;
    // T-segment split (split != 0): the grid holds three roles per (sequence, head)
    float *phi, *psi;             // per pair: segment-1 transition and zero-start state
    __nv_bfloat16 *o_phi;         // [T, H, 128]: segment-1 outputs of the transition run
    int split;
    float *ckpt;                  // chunk-end state checkpoints (backward's forward pass), or null
    uint8_t *fallback;            // per (sequence, head): chain left to the token-sequential kernel, or null
    int prep;                     // input preprocessing flags (PREP_*)
    float prep_eps;               // epsilon of the L2 normalisation
    int64_t T_total, seq_len_fixed;
    int N, H;
    int dk, dv;                   // head dims of the tensors (64 or 128); the tiles are always 128 wide
    float scale;
};

// byte offset of 16-bit element (row, col) in a 128-byte-row tile with the 128B swizzle
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}
__device__ __forceinline__ uint32_t chunk16(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// One m16n8k8 tf32 tile product c += a b (fp32 bit patterns as tf32 operands).
__device__ __forceinline__ void mma_tf32(float (&c)[4], float a0, float a1, float a2, float a3, float b0, float b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(__float_as_uint(a0)), "r"(__float_as_uint(a1)), "r"(__float_as_uint(a2)), "r"(__float_as_uint(a3)),
          "r"(__float_as_uint(b0)), "r"(__float_as_uint(b1)));
}
// Four 8x8 bf16 tiles from shared memory (lanes 8i .. 8i+7 give the row addresses of tile i).
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// One m16n8k16 bf16 tile product c += a b, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packed fp32 pairs: two floats in one 64-bit register pair, multiplied with one
// f32x2 instruction (the decay and state-scaling loops are issue-bound).
__device__ __forceinline__ uint64_t f2(float x, float y) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(x), "f"(y));
    return d;
}
__device__ __forceinline__ float2 uf2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// bf16x2 word -> fp32 pair (exact)
__device__ __forceinline__ uint64_t bf2x(uint32_t w) { return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }
// fp32 pair -> bf16x2 word (round to nearest even)
__device__ __forceinline__ uint32_t pk2(uint64_t v) {
    const float2 f = uf2(v);
    return pack_bf16x2(f.x, f.y);
}
// (x, y) *= (fx, fy) on fp32 bit patterns, one packed multiply
__device__ __forceinline__ void scale2(uint32_t &x, uint32_t &y, float fx, float fy) {
    const float2 t = uf2(mul2(f2(__uint_as_float(x), __uint_as_float(y)), f2(fx, fy)));
    x = __float_as_uint(t.x);
    y = __float_as_uint(t.y);
}
// 2^x (exp(g) is evaluated as 2^(g log2 e))
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// Per-warpgroup register budgets (all four warps of a warpgroup execute the same one).
__device__ __forceinline__ void regs_dec_48() { asm volatile("setmaxnreg.dec.sync.aligned.u32 48;" ::: "memory"); }
__device__ __forceinline__ void regs_inc_120() { asm volatile("setmaxnreg.inc.sync.aligned.u32 120;" ::: "memory"); }
__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

struct Ctl {
    volatile int *abort;
    uint32_t *status;
};

// Bounded wait that also stops early once another role has aborted.
// The waiting thread sleeps inside the barrier probe (up to 20 us at a time), so
// idle roles do not take issue slots from the working ones.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, const Ctl &ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + kWaitNs;
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (*ctl.abort) return false;
        if (globaltimer_ns() > deadline) {
            *ctl.abort = 1;
            atomicOr(ctl.status, DEV_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Wait taken by all threads of a group: every thread waits, then the group
// agrees through a named barrier and its own "first failed wait" index, so either
// all threads go on or all stop (no thread is left alone at a later named
// barrier).  `seq` counts this group's waits identically in every thread.
__device__ __forceinline__ bool group_wait(uint64_t *bar, uint32_t parity, const Ctl &ctl, int *grp_fail, int bar_id,
                                           int nthreads, int &seq) {
    const int w = seq++;
    if (!wait_bar(bar, parity, ctl)) atomicMin(grp_fail, w);
    named_bar(bar_id, nthreads);
    return *reinterpret_cast<volatile int *>(grp_fail) > w;
}

// Wait taken by every lane of a warp, which then agrees on the outcome: all lanes go on or all
// stop.  (Letting lane 0 wait alone while the rest of the warp waits at a shuffle was measured
// markedly slower to resume than this converged wait.)
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const Ctl &ctl) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, ctl)) != 0;
}

// kPrep: the extended instance -- it applies the input preprocessing of p.prep and
// writes the chunk-end checkpoints of p.ckpt (the other instance carries none of that code).
// kNarrow: dk or dv is 64 (p.dk, p.dv); the instances for 128 x 128 heads use the constant
// width, so they carry none of the narrow heads' strides and guards.
template <bool kPrep, bool kNarrow>
__global__ void __launch_bounds__(kThreads, 1) kda_chunk_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t dsmem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(16) float s_beta[2][kC];
    __shared__ __align__(16) float s_ac[3][kD];  // per-chunk A_C, ring of three
    __shared__ __align__(16) float s_x[32 * kLdX];
    __shared__ __align__(16) float s_tot[8][kD];
    __shared__ float s_rn[2][kC];  // inverse L2 norms of this chunk's k and q rows (preprocessing)
    __shared__ uint64_t bar_full[2], bar_free[2];
    __shared__ uint64_t bar_elem, bar_mma1, bar_mfree, bar_tready, bar_mma2, bar_ready, bar_wfree, bar_c1, bar_uready,
        bar_c3;
    __shared__ uint64_t bar_drain[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_grp_fail[3];  // [0] decay group, [1] chain group, [2] solve group

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Without a split, CTA = (sequence, head).  With the T-segment split the full chunks
    // of a sequence are cut in two at a chunk boundary and the grid holds three roles
    // per (sequence, head): 0 = segment 0 from the initial state (normal outputs, state
    // at the cut); 1 = segment 1 from a zero state (its outputs, state Psi); 2 = segment
    // 1 from the identity with v = 0 (outputs Phi_t^T (scale q_t), transition Phi).
    const int64_t npairs = static_cast<int64_t>(p.N) * p.H;
    const int role = p.split ? static_cast<int>(blockIdx.x / npairs) : 0;
    const int64_t slot = p.split ? static_cast<int64_t>(blockIdx.x) % npairs : static_cast<int64_t>(blockIdx.x);
    // with a launch order, consecutive CTAs take the heads of the longest sequences first
    const int64_t pair = p.order ? static_cast<int64_t>(p.order[slot / p.H]) * p.H + slot % p.H : slot;
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    const int64_t H = p.H;

    int64_t bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        bool ok = (bos >= 0) && (bos <= eos) && (eos <= p.T_total);
        if (n == 0 && bos != 0) ok = false;
        if (n == p.N - 1 && eos != p.T_total) ok = false;
        if (!ok) {
            if (tid == 0 && h == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
            return;
        }
    } else {
        bos = static_cast<int64_t>(n) * p.seq_len_fixed;
        eos = bos + p.seq_len_fixed;
    }
    int nfull = static_cast<int>((eos - bos) / kC);  // full chunks of this CTA's segment
    if (p.split) {
        const int n0 = (nfull + 1) / 2;
        if (role == 0) {
            nfull = n0;
        } else {
            bos += static_cast<int64_t>(kC) * n0;
            nfull -= n0;
        }
    }
    if (nfull == 0) return;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_full[s], 2);
            mbar_init(&bar_free[s], 1);
        }
        mbar_init(&bar_elem, 1);
        mbar_init(&bar_mma1, 1);
        mbar_init(&bar_mfree, 1);
        mbar_init(&bar_tready, 1);
        mbar_init(&bar_mma2, 1);
        mbar_init(&bar_ready, 1);
        mbar_init(&bar_wfree, 1);
        mbar_init(&bar_c1, 1);
        mbar_init(&bar_uready, 1);
        mbar_init(&bar_c3, 1);
        mbar_init(&bar_drain[0], 1);
        mbar_init(&bar_drain[1], 1);
        s_abort = 0;
        s_grp_fail[0] = 0x7fffffff;
        s_grp_fail[1] = 0x7fffffff;
        s_grp_fail[2] = 0x7fffffff;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    if (role == 2) {  // the transition run has v = 0: both stages' V tiles stay zero
        for (int i = tid; i < 2 * 16384 / 16; i += kThreads) {
            const int st = i / (16384 / 16), w = i % (16384 / 16);
            reinterpret_cast<uint4 *>(sm + st * kStage + OFF_V)[w] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const Ctl ctl{&s_abort, p.status};
    const uint32_t sm_base = smem_u32(sm);

    // Register split per warpgroup (setmaxnreg; each warpgroup's four warps take the same
    // share): launched with 96 per thread, 61440 for 640 threads (checked on the host);
    // control warps 48, chain and solve groups 120, the two decay warpgroups 96:
    // (48 + 120 + 96 + 96 + 120) x 128 = 61440.
    if (warp < 4) {
        regs_dec_48();
        if (warp == 0) {
            // ------------------------------------------------------------------ TMA producer
            const bool v_zero = (role == 2);
            int issued0 = -1, issued1 = -1;
            for (int c = 0; c < nfull; ++c) {
                const int s = c & 1;
                const int t0 = static_cast<int>(bos + static_cast<int64_t>(c) * kC);
                // beta for this chunk: loaded before waiting for the stage, so its latency overlaps the wait
                float b_lo = __bfloat162float(p.beta[(static_cast<int64_t>(t0) + lane) * H + h]);
                float b_hi = __bfloat162float(p.beta[(static_cast<int64_t>(t0) + lane + 32) * H + h]);
                if constexpr (kPrep) {
                    if (p.prep & PREP_SIGMOID_BETA) {  // beta = sigmoid(x_beta)
                        b_lo = 1.f / (1.f + __expf(-b_lo));
                        b_hi = 1.f / (1.f + __expf(-b_hi));
                    }
                }
                if (c >= 2 && !warp_wait(&bar_free[s], ((c >> 1) - 1) & 1, ctl)) break;
                uint8_t *st = sm + s * kStage;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar_full[s], v_zero ? kStage - 16384 : kStage);
                    tma_load_3d(st + OFF_R + 0, &p.tm_k, 0, h, t0, &bar_full[s]);
                    tma_load_3d(st + OFF_R + 16384, &p.tm_k, 64, h, t0, &bar_full[s]);
                    tma_load_3d(st + OFF_R + 8192, &p.tm_q, 0, h, t0, &bar_full[s]);
                    tma_load_3d(st + OFF_R + 24576, &p.tm_q, 64, h, t0, &bar_full[s]);
                    tma_load_3d(st + OFF_G + 0, &p.tm_g, 0, h, t0, &bar_full[s]);
                    tma_load_3d(st + OFF_G + 8192, &p.tm_g, 64, h, t0, &bar_full[s]);
                    if (!v_zero) {
                        tma_load_3d(st + OFF_V + 0, &p.tm_v, 0, h, t0, &bar_full[s]);
                        tma_load_3d(st + OFF_V + 8192, &p.tm_v, 64, h, t0, &bar_full[s]);
                    }
                    // warm L2 with the chunk that will reuse this stage, so its load is short
                    if (c + 2 < nfull) {
                        const int t2 = t0 + 2 * kC;
                        for (int x = 0; x < 128; x += 64) {  // (boxes beyond dk or dv hold no data)
                            if (!kNarrow || x < p.dk) {
                                tma_prefetch_l2_3d(&p.tm_q, x, h, t2);
                                tma_prefetch_l2_3d(&p.tm_k, x, h, t2);
                                tma_prefetch_l2_3d(&p.tm_g, x, h, t2);
                            }
                            if (!v_zero && (!kNarrow || x < p.dv)) tma_prefetch_l2_3d(&p.tm_v, x, h, t2);
                        }
                    }
                }
                if (s == 0) issued0 = c; else issued1 = c;
                s_beta[s][lane] = b_lo;
                s_beta[s][lane + 32] = b_hi;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_full[s]);
            }
            // make sure no TMA copy is still landing in shared memory when the CTA exits
            const uint64_t deadline = globaltimer_ns() + kWaitNs;
            if (issued0 >= 0)
                while (!mbar_try_wait(&bar_full[0], (issued0 >> 1) & 1) && globaltimer_ns() < deadline) {
                }
            if (issued1 >= 0)
                while (!mbar_try_wait(&bar_full[1], (issued1 >> 1) & 1) && globaltimer_ns() < deadline) {
                }
        } else if (warp == 1) {
            // ------------------------------------------------------------------ chain MMA issuer
            // The whole warp runs this loop and issues through one elected lane (warp-uniform
            // operands: about half the issue time of a branch taken by lane 0 alone).
            {
                const uint32_t idU = idesc_bf16(128, 64, false, true, true);    // U -= S^T W  (W MN-major)
                const uint32_t idO = idesc_bf16(128, 64, false, false);         // O  = S^T Qbar^T, += U^T P^T
                const uint32_t idS = idesc_bf16(128, 128, false, true);         // S += U^T Ktil (Ktil MN-major)
                for (int c = 0; c < nfull; ++c) {
                    const int s = c & 1;
                    if (!warp_wait(&bar_ready, c & 1, ctl)) break;
                    tc_fence_after();
                    const uint32_t st = sm_base + s * kStage;
                    // descriptors built once per chunk; k-steps add constant start offsets
                    const uint64_t dW = sdesc_sw128(st + OFF_R, 8192, 1024);          // W over Kbar, MN-major
                    const uint64_t dQ = sdesc_sw128(st + OFF_R + 8192, 16, 1024);     // Qbar, K-major
                    const uint64_t dP = sdesc_sw128(sm_base + OFF_P + s * 8192, 16, 1024);
                    const uint64_t dG = sdesc_sw128(st + OFF_G, 8192, 1024);          // Ktil, MN-major
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ts_warp(tmem + TM_U, tmem + TM_SB + 8 * ks, dW + (((ks >> 2) * 16384 + (ks & 3) * 2048) >> 4),
                                    idU, 1u);
                    mma_commit_warp(&bar_c1);  // U is on the critical path: release its epilogue first
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ts_warp(tmem + TM_O, tmem + TM_SB + 8 * ks, dQ + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                    idO, ks > 0 ? 1u : 0u);
                    if (!warp_wait(&bar_uready, c & 1, ctl)) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_warp(tmem + TM_S, tmem + TM_UB + 8 * ks, dG + ((ks * 2048) >> 4), idS, 1u);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_warp(tmem + TM_O, tmem + TM_UB + 8 * ks, dP + ((ks * 32) >> 4), idO, 1u);
                    mma_commit_warp(&bar_c3);
                    mma_commit_warp(&bar_free[s]);
                }
                // drain: every MMA the elected lane issued completes before the TMEM is freed
                mma_commit_warp(&bar_drain[0]);
                const uint64_t deadline = globaltimer_ns() + kWaitNs;
                while (!mbar_try_wait(&bar_drain[0], 0) && globaltimer_ns() < deadline) {
                }
            }
        } else if (warp == 2) {
            // ------------------------------------------------------------------ prep MMA issuer
            // Polls both prep MMAs so that the next chunk's [Kbar; Qbar] Ktil^T product can go
            // as soon as its tiles are ready, while this chunk's W / Utl product waits for T'.
            if (lane == 0) {
                const uint32_t id1 = idesc_bf16(128, 64, false, false);  // [Kbar; Qbar] Ktil^T
                const uint32_t id2 = idesc_bf16(128, 64, true, false);   // Kbar^T T'^T, V^T T'^T (A MN-major)
                int c1 = 0, c2 = 0;
                uint64_t deadline = globaltimer_ns() + kWaitNs;
                uint32_t spins = 0;
                while (c2 < nfull) {
                    bool progress = false;
                    if (c1 < nfull && mbar_test_wait(&bar_elem, c1 & 1) &&
                        (c1 == 0 || mbar_test_wait(&bar_mfree, (c1 - 1) & 1))) {
                        tc_fence_after();
                        const uint32_t st = sm_base + (c1 & 1) * kStage;
                        const uint64_t dA = sdesc_sw128(st + OFF_R, 16, 1024);   // [Kbar; Qbar], K-major
                        const uint64_t dB = sdesc_sw128(st + OFF_G, 16, 1024);   // Ktil, K-major
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_bf16_ss(tmem + TM_PREP, dA + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                        dB + (((ks >> 2) * 8192 + (ks & 3) * 32) >> 4), id1, ks > 0 ? 1u : 0u);
                        mma_commit(&bar_mma1);
                        ++c1;
                        progress = true;
                    }
                    if (c2 < c1 && mbar_test_wait(&bar_tready, c2 & 1) &&
                        (c2 == 0 || (mbar_test_wait(&bar_wfree, (c2 - 1) & 1) && mbar_test_wait(&bar_uready, (c2 - 1) & 1)))) {
                        tc_fence_after();
                        const uint32_t st = sm_base + (c2 & 1) * kStage;
                        const uint64_t dK = sdesc_sw128(st + OFF_R, 16384, 1024);  // Kbar^T, MN-major
                        const uint64_t dV = sdesc_sw128(st + OFF_V, 8192, 1024);   // V^T, MN-major
                        const uint64_t dT = sdesc_sw128(sm_base + OFF_TT + (c2 & 1) * 8192, 16, 1024);  // T', K-major
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ss(tmem + TM_W, dK + ((ks * 2048) >> 4), dT + ((ks * 32) >> 4), id2, ks > 0 ? 1u : 0u);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ss(tmem + TM_U, dV + ((ks * 2048) >> 4), dT + ((ks * 32) >> 4), id2, ks > 0 ? 1u : 0u);
                        mma_commit(&bar_mma2);
                        ++c2;
                        progress = true;
                    }
                    if (progress) {
                        deadline = globaltimer_ns() + kWaitNs;
                        spins = 0;
                        continue;
                    }
                    __nanosleep(32);  // back off without stealing issue slots from the math warps
                    if ((++spins & 63u) == 0) {
                        if (*ctl.abort) break;
                        if (globaltimer_ns() > deadline) {
                            *ctl.abort = 1;
                            atomicOr(ctl.status, DEV_ERR_TIMEOUT);
                            break;
                        }
                    }
                }
                mma_commit(&bar_drain[1]);
                const uint64_t dl = globaltimer_ns() + kWaitNs;
                while (!mbar_try_wait(&bar_drain[1], 0) && globaltimer_ns() < dl) {
                }
            }
        }
    } else if (warp < 8) {
        regs_inc_120();
        // ------------------------------------------------------------------ chain group
        const int j = tid - 128;  // TMEM lane: value column j (state, U, O); channel j (W^T)
        int gseq = 0;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + TM_S, tSB = tmem + lane_base + TM_SB;
        // states are dk x dv (row stride dv); channels >= dk and columns >= dv stay zero
        const int sdk = kNarrow ? p.dk : kD, sdv = kNarrow ? p.dv : kD;
        const float *s0 =
            (role == 0 && p.init_state && j < sdv) ? p.init_state + pair * sdk * sdv : nullptr;
        __nv_bfloat16 *const obase = (role == 2) ? p.o_phi : p.o;
        for (int cc = 0; cc < kD; cc += 32) {
            uint32_t a[16], b[16], pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                a[e] = __float_as_uint(s0 && cc + e < sdk ? s0[(cc + e) * sdv + j] : 0.f);
                b[e] = __float_as_uint(s0 && cc + 16 + e < sdk ? s0[(cc + 16 + e) * sdv + j] : 0.f);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                pk[8 + e] = pack_bf16x2(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
            }
            tmem_st16(tS + cc, a);
            tmem_st16(tS + cc + 16, b);
            tmem_st16(tSB + cc / 2, pk);
        }
        if (role == 2) {
            // the transition run starts from the identity: lane j's 1 sits in column j, inside
            // the 32 columns [32 (warp % 4), +32) of its warp
            const int wb = (warp & 3) * 32;
            uint32_t a[16], b[16], pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                a[e] = __float_as_uint(wb + e == j ? 1.f : 0.f);
                b[e] = __float_as_uint(wb + 16 + e == j ? 1.f : 0.f);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                pk[8 + e] = pack_bf16x2(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
            }
            tmem_st_wait();
            tmem_st16(tS + wb, a);
            tmem_st16(tS + wb + 16, b);
            tmem_st16(tSB + wb / 2, pk);
        }
        tmem_st_wait();

        uint32_t opk[32];          // previous chunk's O row block, bf16 pairs (r, r+1)
        int64_t o_t0 = -1;
        auto store_o = [&](int64_t t0) {
            if constexpr (kPrep) {
                if (!obase) return;  // checkpoint-only forward
            }
            if (j >= sdv) return;  // column beyond dv: zero, not stored
            __nv_bfloat16 *orow = obase + (t0 * H + h) * sdv + j;
            const int64_t rs = H * sdv;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&opk[e]);
                orow[(2 * e) * rs] = v.x;
                orow[(2 * e + 1) * rs] = v.y;
            }
        };
        bool done = true;
        for (int c = 0; c < nfull; ++c) {
            const int s = c & 1;
            // W^T (lane = channel) -> bf16 W tile, MN-major (row = channel, 64 tokens)
            if (!group_wait(&bar_mma2, c & 1, ctl, &s_grp_fail[1], 2, 128, gseq)) {
                done = false;
                break;
            }
            tc_fence_after();
            {
                uint8_t *W = sm + s * kStage + OFF_R + (j >> 6) * 16384;  // over Kbar
                const uint32_t tP = tmem + lane_base + TM_W;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t wv[32];
                    tmem_ld16(tP + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&wv[0]));
                    tmem_ld16(tP + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&wv[16]));
                    tmem_ld_wait();
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        uint4 v;
                        uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            vw[e] = pack_bf16x2(__uint_as_float(wv[q8 * 8 + 2 * e]), __uint_as_float(wv[q8 * 8 + 2 * e + 1]));
                        *reinterpret_cast<uint4 *>(W + chunk16(j & 63, 4 * hf + q8)) = v;
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(2, 128);
            if (j == 0) {
                mbar_arrive(&bar_ready);   // W(c) written and the state of chunk c-1 final
                mbar_arrive(&bar_wfree);   // W^T columns may take the next chunk's product
            }
            if (o_t0 >= 0) store_o(o_t0);  // previous chunk's O while C1 runs

            // U (fp32 in TMEM) -> bf16 copy in TMEM, the A operand of P U and Ktil^T U
            if (!group_wait(&bar_c1, c & 1, ctl, &s_grp_fail[1], 2, 128, gseq)) {
                done = false;
                break;
            }
            tc_fence_after();
            {
                const uint32_t tU = tmem + lane_base + TM_U;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t u[32], pk[16];
                    tmem_ld16(tU + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&u[0]));
                    tmem_ld16(tU + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&u[16]));
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1]));
                    tmem_st16(tmem + lane_base + TM_UB + 16 * hf, pk);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            named_bar(2, 128);
            if (j == 0) mbar_arrive(&bar_uready);

            // state: S <- Diag(A_C)(S + Ktil^T U) with its bf16 copy; O into registers
            if (!group_wait(&bar_c3, c & 1, ctl, &s_grp_fail[1], 2, 128, gseq)) {
                done = false;
                break;
            }
            tc_fence_after();
            const bool last = (c == nfull - 1);
            float *sout = (role == 0 ? p.state_out : role == 1 ? p.psi : p.phi) + pair * sdk * sdv;
            for (int cc = 0; cc < kD; cc += 32) {
                uint32_t a[16], b[16], pk[16];
                tmem_ld16(tS + cc, a);
                tmem_ld16(tS + cc + 16, b);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    const float4 fa = ld4(&s_ac[c % 3][cc + e]), fb = ld4(&s_ac[c % 3][cc + 16 + e]);
                    scale2(a[e], a[e + 1], fa.x, fa.y);
                    scale2(a[e + 2], a[e + 3], fa.z, fa.w);
                    scale2(b[e], b[e + 1], fb.x, fb.y);
                    scale2(b[e + 2], b[e + 3], fb.z, fb.w);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                    pk[8 + e] = pack_bf16x2(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
                }
                tmem_st16(tS + cc, a);
                tmem_st16(tS + cc + 16, b);
                tmem_st16(tSB + cc / 2, pk);
                if (last && j < sdv) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (cc + e < sdk) sout[(cc + e) * sdv + j] = __uint_as_float(a[e]);
                        if (cc + 16 + e < sdk) sout[(cc + 16 + e) * sdv + j] = __uint_as_float(b[e]);
                    }
                }
                if constexpr (kPrep) {
                    if (p.ckpt && j < sdv) {  // the state at the start of chunk c + 1 (slot c + 1 of the sequence)
                        float *ck = p.ckpt + ((ckpt_base(bos, n) + c + 1) * H + h) * sdk * sdv;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if (cc + e < sdk) ck[(cc + e) * sdv + j] = __uint_as_float(a[e]);
                            if (cc + 16 + e < sdk) ck[(cc + 16 + e) * sdv + j] = __uint_as_float(b[e]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r0 = 0; r0 < kC; r0 += 32) {
                uint32_t ov[32];
                tmem_ld16(tmem + lane_base + TM_O + r0, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
                tmem_ld16(tmem + lane_base + TM_O + r0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[16]));
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    opk[r0 / 2 + e] = pack_bf16x2(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1]));
            }
            o_t0 = bos + static_cast<int64_t>(c) * kC;
            tmem_st_wait();
            tc_fence_before();
            named_bar(2, 128);
        }
        if (done && o_t0 >= 0) store_o(o_t0);
    } else if (warp >= 8 && warp < 16) {
        // ------------------------------------------------------------------ decay group (warps 8-15)
        // Decay factors and the scaled operand tiles, one chunk ahead of the solve group.
        // Thread = (8-token segment, 4 channels): alpha = exp(g), prefix products within
        // the segment, the earlier segments' totals carried in, then Kbar, Qbar, Ktil
        // written over k, q, g in place.
        const int pt = tid - 256;
        int gseq = 0;
        const float kMinDecay = 7.888609052210118e-31f;  // 2^-100
        for (int c = 0; c < nfull; ++c) {
            const int s = c & 1;
            uint8_t *st = sm + s * kStage;
            if (!group_wait(&bar_full[s], (c >> 1) & 1, ctl, &s_grp_fail[0], 1, 256, gseq)) break;
            {
                // thread = (token segment of 8, channel quad): 64-bit shared accesses
                const int cq = pt & 31, seg = pt >> 5;
                const int kb = cq >> 4, cc = 4 * (cq & 15), ch = kb * 64 + cc;
                uint8_t *Rk = st + OFF_R + kb * 16384;
                uint8_t *Rq = Rk + 8192;
                uint8_t *G = st + OFF_G + kb * 8192;
                const int r0 = 8 * seg;
                uint64_t A01[8], A23[8];
                uint64_t P01 = f2(1.f, 1.f), P23 = f2(1.f, 1.f);
                // Pass 1: running products along the segment.  alpha = exp(g) = 2^(g log2 e),
                // A_r = alpha_1 ... alpha_r.  With the sigmoid gate (preprocessing) alpha =
                // 1 / (1 + 2^(-x log2 e)) and the running product is that of the denominators,
                // D_r = 1 / A_r, so no reciprocal is taken per element here.
                auto pass1 = [&](auto sig) {
                    constexpr bool kSig = decltype(sig)::value;
                    const float l2e = kSig ? -1.4426950408889634f : 1.4426950408889634f;
                    const uint64_t L2E = f2(l2e, l2e);
#pragma unroll
                    for (int rr = 0; rr < 8; rr += 4) {
                        uint2 gw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) gw[e] = *reinterpret_cast<const uint2 *>(G + swz(r0 + rr + e, cc));
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 l01 = uf2(mul2(bf2x(gw[e].x), L2E)), l23 = uf2(mul2(bf2x(gw[e].y), L2E));
                            const uint64_t e01 = f2(ex2_approx(l01.x), ex2_approx(l01.y));
                            const uint64_t e23 = f2(ex2_approx(l23.x), ex2_approx(l23.y));
                            if constexpr (kSig) {
                                P01 = fma2(P01, e01, P01);  // D *= 1 + e
                                P23 = fma2(P23, e23, P23);
                            } else {
                                P01 = mul2(P01, e01);
                                P23 = mul2(P23, e23);
                            }
                            A01[rr + e] = P01;
                            A23[rr + e] = P23;
                        }
                    }
                };
                bool sig_gate = false, norms = false;
                if constexpr (kPrep) {
                    sig_gate = (p.prep & PREP_SIGMOID_GATE) != 0;
                    norms = (p.prep & (PREP_L2NORM_K | PREP_L2NORM_Q)) != 0;
                }
                // Row norms (preprocessing): each of the eight warps takes one 16-row block of k
                // (warps 0-3) or q (warps 4-7) and forms the diagonal of its Gram block with
                // m16n8k16 tensor-core tiles: a 16 x 16 slice loaded by ldmatrix is the A operand
                // and, for each 8-row half, the B operand.  Issued before the first pass so that
                // their latency overlaps it.
                float nc0[4] = {0.f, 0.f, 0.f, 0.f}, nc1[4] = {0.f, 0.f, 0.f, 0.f};
                const int ntq = seg >> 2, nblk = seg & 3;
                if constexpr (kPrep) {
                    if (norms) {
                        const uint32_t nbase = sm_base + s * kStage + OFF_R + ntq * 8192;
                        const int nrow = 16 * nblk + (cq & 7) + ((cq >> 3) & 1) * 8;
#pragma unroll
                        for (int nk = 0; nk < 8; ++nk) {
                            uint32_t fa[4];
                            ldmatrix_x4(fa, nbase + (nk >> 2) * 16384 + chunk16(nrow, 2 * (nk & 3) + (cq >> 4)));
                            mma_bf16_16816(nc0, fa, fa[0], fa[2]);  // block x its rows 0-7
                            mma_bf16_16816(nc1, fa, fa[1], fa[3]);  // block x its rows 8-15
                        }
                    }
                }
                if (sig_gate)
                    pass1(std::true_type{});
                else
                    pass1(std::false_type{});
                if constexpr (kPrep) {
                    // lane (g, g / 2) of the m16n8 accumulator layout holds rows g and g + 8 of the diagonal
                    const int g8 = cq >> 2;
                    if (norms && (cq & 3) == (g8 >> 1)) {
                        const bool on = (p.prep & (ntq == 0 ? PREP_L2NORM_K : PREP_L2NORM_Q)) != 0;
                        const float lo = (g8 & 1) ? nc0[1] : nc0[0], hi = (g8 & 1) ? nc1[3] : nc1[2];
                        s_rn[ntq][16 * nblk + g8] = on ? rsqrtf(lo + p.prep_eps) : 1.f;
                        s_rn[ntq][16 * nblk + g8 + 8] = on ? rsqrtf(hi + p.prep_eps) : 1.f;
                    }
                }
                const float2 pp01 = uf2(P01), pp23 = uf2(P23);
                const float p0 = pp01.x, p1 = pp01.y, p2 = pp23.x, p3 = pp23.y;
                st4(&s_tot[seg][ch], make_float4(p0, p1, p2, p3));
                named_bar(1, 256);
                float4 m = make_float4(1.f, 1.f, 1.f, 1.f);  // product of the earlier segments' totals
                for (int q = 0; q < seg; ++q) {
                    const float4 t = ld4(&s_tot[q][ch]);
                    m = make_float4(m.x * t.x, m.y * t.y, m.z * t.z, m.w * t.w);
                }
                const float sc = p.scale;
                const uint64_t m01 = f2(m.x, m.y), m23 = f2(m.z, m.w);
                const uint64_t ms01 = f2(m.x * sc, m.y * sc), ms23 = f2(m.z * sc, m.w * sc);
                // Pass 2: Kbar = k A, Qbar = scale q A, Ktil = k / A over k, q, g in place.  With
                // L2-normalised rows (preprocessing) k and q are first scaled by their rows'
                // inverse norms; with the sigmoid gate the running products are D = 1 / A.
                auto pass2 = [&](auto norm, auto sig) {
                    constexpr bool kNorm = decltype(norm)::value;
                    constexpr bool kSig = decltype(sig)::value;
#pragma unroll
                    for (int rr = 0; rr < 8; rr += 2) {
                        uint2 kw[2], qw[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t off = swz(r0 + rr + e, cc);
                            kw[e] = *reinterpret_cast<const uint2 *>(Rk + off);
                            qw[e] = *reinterpret_cast<const uint2 *>(Rq + off);
                        }
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t off = swz(r0 + rr + e, cc);
                            uint64_t a01, a23, aq01, aq23, r01, r23;
                            if constexpr (kSig) {
                                r01 = mul2(m01, A01[rr + e]);
                                r23 = mul2(m23, A23[rr + e]);
                                const float2 fr01 = uf2(r01), fr23 = uf2(r23);
                                a01 = f2(rcp_approx(fr01.x), rcp_approx(fr01.y));
                                a23 = f2(rcp_approx(fr23.x), rcp_approx(fr23.y));
                                aq01 = mul2(a01, f2(sc, sc));
                                aq23 = mul2(a23, f2(sc, sc));
                            } else {
                                a01 = mul2(m01, A01[rr + e]);
                                a23 = mul2(m23, A23[rr + e]);
                                aq01 = mul2(ms01, A01[rr + e]);
                                aq23 = mul2(ms23, A23[rr + e]);
                                const float2 fa01 = uf2(a01), fa23 = uf2(a23);
                                r01 = f2(rcp_approx(fa01.x), rcp_approx(fa01.y));
                                r23 = f2(rcp_approx(fa23.x), rcp_approx(fa23.y));
                            }
                            uint64_t k01 = bf2x(kw[e].x), k23 = bf2x(kw[e].y);
                            uint64_t q01 = bf2x(qw[e].x), q23 = bf2x(qw[e].y);
                            if constexpr (kNorm) {
                                const float rk = s_rn[0][r0 + rr + e], rq = s_rn[1][r0 + rr + e];
                                k01 = mul2(k01, f2(rk, rk));
                                k23 = mul2(k23, f2(rk, rk));
                                q01 = mul2(q01, f2(rq, rq));
                                q23 = mul2(q23, f2(rq, rq));
                            }
                            *reinterpret_cast<uint2 *>(Rk + off) = make_uint2(pk2(mul2(k01, a01)), pk2(mul2(k23, a23)));
                            *reinterpret_cast<uint2 *>(Rq + off) = make_uint2(pk2(mul2(q01, aq01)), pk2(mul2(q23, aq23)));
                            *reinterpret_cast<uint2 *>(G + off) = make_uint2(pk2(mul2(k01, r01)), pk2(mul2(k23, r23)));
                        }
                    }
                };
                float4 ac;  // A_C of the chunk (segment 7 holds the last products)
                if constexpr (!kPrep) {
                    pass2(std::false_type{}, std::false_type{});
                    ac = make_float4(m.x * p0, m.y * p1, m.z * p2, m.w * p3);
                } else {
                    if (norms) {
                        if (sig_gate) pass2(std::true_type{}, std::true_type{});
                        else pass2(std::true_type{}, std::false_type{});
                    } else {
                        if (sig_gate) pass2(std::false_type{}, std::true_type{});
                        else pass2(std::false_type{}, std::false_type{});
                    }
                    const float4 x = make_float4(m.x * p0, m.y * p1, m.z * p2, m.w * p3);
                    ac = sig_gate ? make_float4(rcp_approx(x.x), rcp_approx(x.y), rcp_approx(x.z), rcp_approx(x.w)) : x;
                }
                if (seg == 7) {
                    if (!(ac.x >= kMinDecay) || !(ac.y >= kMinDecay) || !(ac.z >= kMinDecay) || !(ac.w >= kMinDecay)) {
                        // out of the factored form's range: the token-sequential kernel redoes the chain
                        // (its results here are discarded), or, without room for that flag, an error
                        if (p.fallback)
                            p.fallback[pair] = 1;
                        else
                            atomicOr(p.status, DEV_ERR_GATE);
                    }
                    st4(&s_ac[c % 3][ch], ac);
                }
            }
            fence_proxy_async_smem();
            named_bar(1, 256);
            if (pt == 0) {
                // at most one chunk ahead of the MMA that consumes these tiles
                if (c > 0) wait_bar(&bar_mma1, (c - 1) & 1, ctl);
                mbar_arrive(&bar_elem);
            }
        }
    } else if (warp >= 16) {
        regs_inc_120();
        // ------------------------------------------------------------------ solve group (warps 16-19)
        const int pt = tid - 512;
        const int wq = warp & 3;
        int gseq = 0;
        float *Mb = reinterpret_cast<float *>(sm + OFF_M);
        float *Tb = reinterpret_cast<float *>(sm + OFF_T);
        for (int i = pt; i < 64 * kLdT; i += 128) Tb[i] = 0.f;  // blocks above the diagonal stay zero
        for (int i = pt; i < 2 * 8192 / 16; i += 128) {         // likewise in both T' tiles; both P tiles
            reinterpret_cast<uint4 *>(sm + OFF_TT)[i] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4 *>(sm + OFF_P)[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        named_bar(3, 128);
        for (int c = 0; c < nfull; ++c) {
            const int s = c & 1;
            uint8_t *TT = sm + OFF_TT + (c & 1) * 8192;  // this chunk's T' = T Diag(beta), bf16
            // (2) M (fp32, rows scaled by beta, strictly lower) and P (bf16, lower incl.).
            // Accumulator lane x: rows 0-63 = Kbar . Ktil, 64-127 = Qbar . Ktil.
            if (!group_wait(&bar_mma1, c & 1, ctl, &s_grp_fail[2], 3, 128, gseq)) break;
            tc_fence_after();
            {
                // Warps 0 / 2 of the group hold rows 0-31 of M / P, which need only columns 0-31
                // (M is read strictly below the diagonal; P's columns 32-63 there stay zero).
                const int x = wq * 32 + lane;
                const bool low = (wq & 1) == 0;
                uint32_t m[64];
                const uint32_t tP = tmem + (static_cast<uint32_t>(wq * 32) << 16) + TM_PREP;
                tmem_ld16(tP + 0, *reinterpret_cast<uint32_t(*)[16]>(&m[0]));
                tmem_ld16(tP + 16, *reinterpret_cast<uint32_t(*)[16]>(&m[16]));
                if (!low) {
                    tmem_ld16(tP + 32, *reinterpret_cast<uint32_t(*)[16]>(&m[32]));
                    tmem_ld16(tP + 48, *reinterpret_cast<uint32_t(*)[16]>(&m[48]));
                }
                tmem_ld_wait();
                if (x < 64) {
                    // M = beta_r (Kbar Ktil^T)[r, :]; entries on and above the diagonal are never read
                    const int r = x;
                    const uint64_t b2 = f2(s_beta[s][r], s_beta[s][r]);
                    float *row = &Mb[r * kLdM];
                    auto put4 = [&](int i) {
                        const float2 u = uf2(mul2(f2(__uint_as_float(m[i]), __uint_as_float(m[i + 1])), b2));
                        const float2 w = uf2(mul2(f2(__uint_as_float(m[i + 2]), __uint_as_float(m[i + 3])), b2));
                        st4(row + i, make_float4(u.x, u.y, w.x, w.y));
                    };
#pragma unroll
                    for (int i = 0; i < 32; i += 4) put4(i);
                    if (!low) {
#pragma unroll
                        for (int i = 32; i < 64; i += 4) put4(i);
                    }
                } else {
                    // P = (Qbar Ktil^T)[r, :] for i <= r, bf16
                    const int r = x - 64;
                    uint8_t *P = sm + OFF_P + s * 8192;
                    auto put8 = [&](int q8, bool masked) {
                        uint4 v;
                        uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = q8 * 8 + 2 * e;
                            const float x0 = (!masked || i0 <= r) ? __uint_as_float(m[i0]) : 0.f;
                            const float x1 = (!masked || i0 + 1 <= r) ? __uint_as_float(m[i0 + 1]) : 0.f;
                            vw[e] = pack_bf16x2(x0, x1);
                        }
                        *reinterpret_cast<uint4 *>(P + chunk16(r, q8)) = v;
                    };
                    if (low) {
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) put8(q8, true);
                    } else {
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) put8(q8, false);
#pragma unroll
                        for (int q8 = 4; q8 < 8; ++q8) put8(q8, true);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(3, 128);
            if (pt == 0) mbar_arrive(&bar_mfree);  // PREP columns may take the next chunk's product

            // (3) T = (I + M)^-1, blocked: the four 16x16 diagonal blocks D_b by forward
            // substitution, column-oriented (warp = block, lane = column, so the four blocks run
            // on all four schedulers; each solved entry is pushed into every later row at once;
            // M read four columns at a time) ...
            if (lane < 16) {
                const int b = wq, mm = lane, R0 = 16 * b;
                float acc[16], xv[16];
#pragma unroll
                for (int l = 0; l < 16; ++l) acc[l] = 0.f;
#pragma unroll
                for (int i0 = 0; i0 < 16; i0 += 4) {
                    float4 mq[16];
#pragma unroll
                    for (int l = i0 + 1; l < 16; ++l) mq[l] = ld4(&Mb[(R0 + l) * kLdM + R0 + i0]);
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const int i = i0 + ii;
                        xv[i] = (i < mm) ? 0.f : ((i == mm) ? 1.f : -acc[i]);
#pragma unroll
                        for (int l = i + 1; l < 16; ++l) {
                            const float mv = ii == 0 ? mq[l].x : ii == 1 ? mq[l].y : ii == 2 ? mq[l].z : mq[l].w;
                            acc[l] = fmaf(mv, xv[i], acc[l]);
                        }
                    }
                }
                const float bm = s_beta[s][R0 + mm];
#pragma unroll
                for (int l = 0; l < 16; ++l) {
                    Tb[(R0 + l) * kLdT + R0 + mm] = xv[l];
                    *reinterpret_cast<__nv_bfloat16 *>(TT + swz(R0 + l, R0 + mm)) = __float2bfloat16_rn(xv[l] * bm);
                }
            }
            named_bar(3, 128);
            // ... then the off-diagonal blocks as tf32 tensor-core tiles (m16n8k8; each warp
            // owns output tiles): fragment row gq = lane / 4, column tq = lane % 4.
            const int gq = lane >> 2, tq = lane & 3;
            {
                // sub-diagonal blocks T[a][a-1] = -D_a (M[a][a-1] D_{a-1}), a = 1 (warps 0,1), 3 (warps 2,3)
                const int pr = wq >> 1, nt = wq & 1;
                const int Ra = 16 + 32 * pr, Rb = Ra - 16, n0 = 8 * nt;
                float *X = s_x + pr * 16 * kLdX;
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = 8 * ks;
                    mma_tf32(c, Mb[(Ra + gq) * kLdM + Rb + k0 + tq], Mb[(Ra + gq + 8) * kLdM + Rb + k0 + tq],
                             Mb[(Ra + gq) * kLdM + Rb + k0 + tq + 4], Mb[(Ra + gq + 8) * kLdM + Rb + k0 + tq + 4],
                             Tb[(Rb + k0 + tq) * kLdT + Rb + n0 + gq], Tb[(Rb + k0 + tq + 4) * kLdT + Rb + n0 + gq]);
                }
                X[gq * kLdX + n0 + 2 * tq] = c[0];
                X[gq * kLdX + n0 + 2 * tq + 1] = c[1];
                X[(gq + 8) * kLdX + n0 + 2 * tq] = c[2];
                X[(gq + 8) * kLdX + n0 + 2 * tq + 1] = c[3];
                named_bar(3, 128);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = 8 * ks;
                    mma_tf32(d, Tb[(Ra + gq) * kLdT + Ra + k0 + tq], Tb[(Ra + gq + 8) * kLdT + Ra + k0 + tq],
                             Tb[(Ra + gq) * kLdT + Ra + k0 + tq + 4], Tb[(Ra + gq + 8) * kLdT + Ra + k0 + tq + 4],
                             X[(k0 + tq) * kLdX + n0 + gq], X[(k0 + tq + 4) * kLdX + n0 + gq]);
                }
                const int cl = Rb + n0 + 2 * tq;
                Tb[(Ra + gq) * kLdT + cl] = -d[0];
                Tb[(Ra + gq) * kLdT + cl + 1] = -d[1];
                Tb[(Ra + gq + 8) * kLdT + cl] = -d[2];
                Tb[(Ra + gq + 8) * kLdT + cl + 1] = -d[3];
                const float b0 = s_beta[s][cl], b1 = s_beta[s][cl + 1];
                *reinterpret_cast<uint32_t *>(TT + swz(Ra + gq, cl)) = pack_bf16x2(-d[0] * b0, -d[1] * b1);
                *reinterpret_cast<uint32_t *>(TT + swz(Ra + gq + 8, cl)) = pack_bf16x2(-d[2] * b0, -d[3] * b1);
            }
            named_bar(3, 128);
            {
                // lower-left quadrant T[32:64, 0:32] = -T22 (M[32:64, 0:32] T11); T11 = T[0:32, 0:32],
                // T22 = T[32:64, 32:64] (their upper-right blocks are zero).  Warp: 16 rows x 16 cols.
                const int mt = wq >> 1, nh = wq & 1;
                const int r0 = 16 * mt;
                float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const int k0 = 8 * ks;
                    const float a0 = Mb[(32 + r0 + gq) * kLdM + k0 + tq], a1 = Mb[(40 + r0 + gq) * kLdM + k0 + tq];
                    const float a2 = Mb[(32 + r0 + gq) * kLdM + k0 + tq + 4], a3 = Mb[(40 + r0 + gq) * kLdM + k0 + tq + 4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int n0 = 16 * nh + 8 * nt;
                        mma_tf32(c[nt], a0, a1, a2, a3, Tb[(k0 + tq) * kLdT + n0 + gq], Tb[(k0 + tq + 4) * kLdT + n0 + gq]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int n0 = 16 * nh + 8 * nt;
                    s_x[(r0 + gq) * kLdX + n0 + 2 * tq] = c[nt][0];
                    s_x[(r0 + gq) * kLdX + n0 + 2 * tq + 1] = c[nt][1];
                    s_x[(r0 + gq + 8) * kLdX + n0 + 2 * tq] = c[nt][2];
                    s_x[(r0 + gq + 8) * kLdX + n0 + 2 * tq + 1] = c[nt][3];
                }
                named_bar(3, 128);
                float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const int k0 = 8 * ks;
                    const float a0 = Tb[(32 + r0 + gq) * kLdT + 32 + k0 + tq], a1 = Tb[(40 + r0 + gq) * kLdT + 32 + k0 + tq];
                    const float a2 = Tb[(32 + r0 + gq) * kLdT + 36 + k0 + tq], a3 = Tb[(40 + r0 + gq) * kLdT + 36 + k0 + tq];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int n0 = 16 * nh + 8 * nt;
                        mma_tf32(d[nt], a0, a1, a2, a3, s_x[(k0 + tq) * kLdX + n0 + gq], s_x[(k0 + tq + 4) * kLdX + n0 + gq]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int cl = 16 * nh + 8 * nt + 2 * tq;
                    const float b0 = s_beta[s][cl], b1 = s_beta[s][cl + 1];
                    *reinterpret_cast<uint32_t *>(TT + swz(32 + r0 + gq, cl)) =
                        pack_bf16x2(-d[nt][0] * b0, -d[nt][1] * b1);
                    *reinterpret_cast<uint32_t *>(TT + swz(40 + r0 + gq, cl)) =
                        pack_bf16x2(-d[nt][2] * b0, -d[nt][3] * b1);
                }
            }
            // T' was written block by block above (its tile's previous content, chunk c-2,
            // was consumed before the previous chunk announced its T').  Announce this
            // chunk's T' only once the previous chunk's W / Utl product has completed: that
            // product consumed the previous announcement, so the barrier phases cannot alias.
            if (c > 0 && !group_wait(&bar_mma2, (c - 1) & 1, ctl, &s_grp_fail[2], 3, 128, gseq)) break;
            fence_proxy_async_smem();
            named_bar(3, 128);
            if (pt == 0) mbar_arrive(&bar_tready);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [T, H, D] bf16 tensor (D = 64 or 128), 64 x 64 boxes with the 128-byte swizzle.  The kernel
// reads channels [0, 128) in two boxes; with D = 64 the second box lies wholly beyond the
// tensor and arrives as zeros (its x coordinate, 64, keeps the 16-byte rule).
bool encode_tile_map(CUtensorMap *map, const void *base, int64_t T, int H, int D) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {
// order[rank] = n: rank = sequences with more full chunks, or as many and a lower index.
__global__ void __launch_bounds__(256) order_kernel(const int32_t *cu, int N, int32_t *order) {
    const int n = static_cast<int>(blockIdx.x) * 256 + static_cast<int>(threadIdx.x);
    if (n >= N) return;
    const int64_t cn = (static_cast<int64_t>(cu[n + 1]) - cu[n]) / kC;
    int r = 0;
    for (int m = 0; m < N; ++m) {
        const int64_t cm = (static_cast<int64_t>(cu[m + 1]) - cu[m]) / kC;
        r += (cm > cn || (cm == cn && m < n)) ? 1 : 0;
    }
    order[r] = n;
}
}  // namespace

cudaError_t launch_order(const int32_t *cu, int N, int32_t *order, cudaStream_t stream) {
    if (N <= 0) return cudaSuccess;
    order_kernel<<<static_cast<unsigned>((N + 255) / 256), 256, 0, stream>>>(cu, N, order);
    return cudaGetLastError();
}

bool chunk_tc_supported(int dk, int dv, int dtype) {
    return (dk == 64 || dk == 128) && (dv == 64 || dv == 128) && dtype == 0;
}

cudaError_t launch_chunk_tc(const ChunkParams &cp, cudaStream_t stream) {
    const int dk = cp.dk ? cp.dk : kD, dv = cp.dv ? cp.dv : kD;
    if (!chunk_tc_supported(dk, dv, 0)) return cudaErrorNotSupported;
    // the T-segment roles and their merge are laid out 128 x 128
    if (cp.split && (dk != kD || dv != kD)) return cudaErrorNotSupported;
    const int64_t seqs = (cp.order && !cp.split) ? cp.n_active : cp.N;
    const int64_t blocks = seqs * cp.H * (cp.split ? 3 : 1);
    if (blocks <= 0 || cp.T_total <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    TcParams p{};
    if (!encode_tile_map(&p.tm_q, cp.q, cp.T_total, cp.H, dk) || !encode_tile_map(&p.tm_k, cp.k, cp.T_total, cp.H, dk) ||
        !encode_tile_map(&p.tm_g, cp.g, cp.T_total, cp.H, dk) || !encode_tile_map(&p.tm_v, cp.v, cp.T_total, cp.H, dv))
        return cudaErrorInvalidValue;
    p.dk = dk;
    p.dv = dv;
    p.beta = static_cast<const __nv_bfloat16 *>(cp.beta);
    p.o = static_cast<__nv_bfloat16 *>(cp.o);
    p.cu = cp.cu;
    p.init_state = cp.init_state;
    p.state_out = cp.state_out;
    p.status = cp.status;
    p.T_total = cp.T_total;
    p.seq_len_fixed = cp.seq_len_fixed;
    p.N = cp.N;
    p.H = cp.H;
    p.scale = cp.scale;
    p.split = cp.split;
    p.prep = cp.prep;
    p.prep_eps = cp.prep_eps;
    p.phi = cp.phi;
    p.psi = cp.psi;
    p.o_phi = static_cast<__nv_bfloat16 *>(cp.o_phi);
    p.ckpt = cp.ckpt;
    p.fallback = cp.fallback;
    p.order = cp.split ? nullptr : cp.order;
    // The register split assumes 96 registers per thread at launch (a property of the compiled
    // image, checked once).  The dynamic shared-memory limit is a function attribute of the device
    // that is current when it is set, so it is set on every launch (a host-side call that
    // allocates nothing and does not synchronize).
    static std::atomic<int> regs_ok{0};  // 0 unknown, 1 as assumed, 2 not
    for (auto fn : {kda_chunk_tc_kernel<false, false>, kda_chunk_tc_kernel<true, false>,
                    kda_chunk_tc_kernel<false, true>, kda_chunk_tc_kernel<true, true>}) {
        if (regs_ok.load(std::memory_order_acquire) == 0) {
            cudaFuncAttributes fa{};
            if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return cudaErrorInvalidConfiguration;
            if (fa.numRegs != 96) regs_ok.store(2, std::memory_order_release);
        }
        if (regs_ok.load(std::memory_order_acquire) == 2) return cudaErrorInvalidConfiguration;
        const cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kDynSmem));
        if (e != cudaSuccess) return e;
    }
    int unknown = 0;
    regs_ok.compare_exchange_strong(unknown, 1);
    const unsigned grid = static_cast<unsigned>(blocks);
    const bool ext = p.prep || p.ckpt, narrow = dk != kD || dv != kD;
    if (narrow) {
        if (ext) kda_chunk_tc_kernel<true, true><<<grid, kThreads, kDynSmem, stream>>>(p);
        else kda_chunk_tc_kernel<false, true><<<grid, kThreads, kDynSmem, stream>>>(p);
    } else {
        if (ext) kda_chunk_tc_kernel<true, false><<<grid, kThreads, kDynSmem, stream>>>(p);
        else kda_chunk_tc_kernel<false, false><<<grid, kThreads, kDynSmem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
