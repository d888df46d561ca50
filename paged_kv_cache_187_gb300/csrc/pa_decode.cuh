// pa_decode.cuh -- the paged decode-attention kernel for sm_103a.
//
// What it computes ("vLLM Project Update" talk, parts on PagedAttention and on the V2
// kernel; "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention" thread, exact
// attention): for each sequence s and query head h,
//     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) v_t,   t < context_len[s],
// where token t lives in row t % block_size of physical block block_tables[s][t / bs],
// kv head h / group.  A work unit is (sequence, kv head, token range): the whole
// context (V1) or one partition of partition_size tokens (V2); multi-query units also
// carry a chunk of the (query token, head) rows.  A V2 unit of a sequence
// with several partitions stores its partial (max, exp-sum, unnormalised sum); the last
// unit of that (sequence, kv head) to finish merges all partials by log-sum-exp, so no
// separate reduction launch is needed.
//
// GB300 design (one CTA = 1 producer warp + NCONS consumer warps, several CTAs per SM):
//   * the producer takes work units, copies the unit's query rows with a 1-D bulk copy,
//     and streams the unit's K and V tiles -- a (block, kv head) box is block_size x
//     head_size contiguous elements; an fp8 tile over 16-token blocks holds two -- with
//     2-D tensor TMA into an NSTAGE-deep ring of shared-memory stages (128-byte swizzle,
//     L2 evict-first);
//   * the consumers take the tiles round robin and run the online softmax over them; at
//     the end of a unit the consumer of its last tile merges the others' states (through
//     shared memory) and writes the result while the others start the next unit:
//       - group >= 2 (GQA), and fp8 caches: S^T = K_tile Q^T and O^T += V_tile^T P^T on
//         the tensor cores (mma.sync m16n8k16, tokens / head dims on M, the group's
//         query heads on N), P moved from accumulator to operand layout with movmatrix;
//         fp8 tiles are widened to fp16 fragments in registers;
//       - group 1 (MHA) over a 16-bit cache, or on request: CUDA cores, each lane owning
//         head_size/32 dims, dot products finished by a transposed butterfly reduction;
//       - several query tokens per sequence (multi-query, to verify speculative
//         tokens): the tensor-core path with (query token, head) pairs on N, each
//         column masked causally at its own token limit;
//   * all barrier waits are bounded; a timeout is reported, never hung on.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

#define PA_DEVERR_BAD_BLOCK_ 2
#define PA_DEVERR_BAD_LEN_ 4
#define PA_DEVERR_TIMEOUT_ 8

// Tiles of the current unit still to issue when the producer claims the next unit.
#ifndef PA_CLAIM_LEAD
#define PA_CLAIM_LEAD 8
#endif

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^(m - M) with the convention that an empty state (m = -inf) weighs 0.
__device__ __forceinline__ float state_weight(float m, float M) {
    return m == -INFINITY ? 0.f : fast_exp2(m - M);
}

__device__ __forceinline__ void flag_error(int32_t* status, int32_t bit) {
    if (status) atomicOr(status, bit);
}

// Context length of sequence s, clamped to what the host promised and the block-table
// row can hold.  Every kernel uses this same clamp so their views of a unit agree.
__device__ __forceinline__ int32_t clamped_len(const DecodeParams& p, int32_t s, bool report) {
    int32_t L = p.context_lens[s];
    const int64_t row_cap = (int64_t)p.max_blocks_per_seq * p.block_size;
    const int32_t cap = row_cap < p.max_context_len ? (int32_t)row_cap : p.max_context_len;
    if (L < 0 || L > cap) {
        if (report) flag_error(p.status, PA_DEVERR_BAD_LEN_);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// Named barrier `bar` (1 unless a kernel has several groups of consumer warps) among the
// consumer warps only (the producer never joins it) that also ORs a flag over every
// consumer thread, so all consumers take the same branch.
__device__ __forceinline__ bool consumers_any(bool v, int nthreads, int bar = 1) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %3, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(nthreads), "r"(bar)
        : "memory");
    return r != 0;
}

// A bounded barrier wait whose result is the same in every lane of the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// Is the CTA aborting?  The same answer in every lane of the warp.
__device__ __forceinline__ bool warp_sees_abort(const volatile int32_t& flag) {
    return __any_sync(0xffffffffu, flag != 0);
}

struct UnitDesc {
    int32_t seq;     // -1: no more units
    int32_t kvh;
    int32_t tok0;    // first token of the unit (a multiple of block_size)
    int32_t tok1;    // one past the last token
    int32_t pslot;   // partition slot for partial results, -1: write the final output
    int32_t pbase;   // first partition slot of the sequence
    int32_t nparts;  // partitions of the sequence
    int32_t row0;    // first query row of the unit (rows: see DecodeParams)
    int32_t nrows;   // query rows of the unit
    int32_t len;     // context length of the sequence (multi-query causal limits)
    int32_t pad[2];
};

template <int D_, int BS_, bool BF16_, bool MMA_, int HCAP_, int NSTAGE_, int NQ_, int NCONS_,
          bool KV8_ = false, bool MQ_ = false, int MINB_ = 0, int PBS_ = BS_>
struct DecodeCfg {
    static constexpr int D = D_;
    // Tokens per tile (what a consumer takes at a time), and the pool's block size: a tile
    // is TB = BS / PBS consecutive blocks of the sequence, gathered into one stage.
    static constexpr int BS = BS_;
    static constexpr int PBS = PBS_;
    static constexpr int TB = BS_ / PBS_;
    static constexpr bool kBf16 = BF16_;           // query / output type (bf16 or fp16)
    static constexpr bool kKv8 = KV8_;             // K/V cache in fp8 E4M3 (else = query type)
    static constexpr bool kMma = MMA_;
    static constexpr bool kMq = MQ_;               // several causal query tokens per sequence
    static constexpr int HCAP = HCAP_;             // query rows per unit the kernel holds
    static constexpr int NT = MMA_ ? HCAP_ / 8 : 0;  // mma n-tiles of 8 heads
    static constexpr int NSTAGE = NSTAGE_;
    static constexpr int NQ = NQ_;
    static constexpr int NCONS = NCONS_;           // consumer warps per CTA
    static constexpr int ELEM = KV8_ ? 1 : 2;      // bytes per cached element
    static constexpr int HALVES = D * ELEM / 128;  // 128-byte swizzle spans per row
    static constexpr int TILE_BYTES = D * BS * ELEM;  // one tile of K or V (one kv head)
    static constexpr int HALF_BYTES = BS * 128;
    // multi-query: a unit has up to NCONS row groups of HCAP rows, each finished by its
    // own consumer
    static constexpr int QROWS = (MQ_ ? NCONS_ : 1) * HCAP;
    static constexpr int THREADS = 32 * (1 + NCONS);
    // Resident CTAs per SM the register allocation is sized for; 0 leaves the choice to
    // the compiler (see decode_min_ctas).
    static constexpr int MIN_CTAS = MINB_;
    // per-lane floats of one consumer's softmax state (m, l, acc)
    static constexpr int NSTATE = MMA_ ? (4 * NT + (D / 16) * NT * 4) : (2 * HCAP_ + HCAP_ * (D / 32));
    static_assert(D == 64 || D == 128, "head_size");
    static_assert(BS == 16 || BS == 32, "tile tokens");
    static_assert((PBS_ == 16 || PBS_ == 32) && BS_ % PBS_ == 0, "block_size");
    static_assert(!MMA_ || HCAP_ == 8 || HCAP_ == 16, "mma heads");
    static_assert(MMA_ || HCAP_ == 1 || HCAP_ == 2 || HCAP_ == 4 || HCAP_ == 8, "heads");
    static_assert(NCONS >= 1 && NCONS <= 4, "consumers");
    // Tile k (counted over all units) goes to consumer k % NCONS (of its row group) and
    // lands in stage k % NSTAGE.  With NSTAGE a multiple of NCONS, the previous use of a
    // stage (tile k - NSTAGE) belongs to the same consumer, so a consumer never waits on
    // a stage that is two phases behind -- where the mbarrier parity test would pass too
    // early.
    static_assert(NSTAGE % NCONS == 0, "stages must be a multiple of the consumer warps");
    static_assert(!KV8_ || D == 128, "fp8 K/V: head_size 128");
    static_assert(!MQ_ || (MMA_ && !KV8_), "multi-query: tensor-core path, 16-bit cache");
};

template <class C>
struct alignas(1024) DecodeSmem {
    uint8_t kv[C::NSTAGE][2][C::TILE_BYTES];         // stage: K tile then V tile
    alignas(128) uint8_t qbuf[C::NQ][C::QROWS * C::D * 2];
    // Output staging of a unit's leader.  Multi-query kernels stage each row group's
    // output in one of the group's state slots instead (see the consumer loop).
    alignas(128) float ostage[C::kMq ? 1 : C::HCAP * C::D];
    // State slots: the consumers other than a unit's leader export their softmax states
    // here for merging (NCONS - 1 slots); multi-query kernels have one slot per consumer.
    alignas(16) float xbuf[C::kMq ? C::NCONS : (C::NCONS > 1 ? C::NCONS - 1 : 1)][C::NSTATE * 32];
    // CUDA-core path: softmax weights
    alignas(16) float pbuf[C::kMma ? 1 : C::NCONS][C::kMma ? 1 : C::HCAP][C::kMma ? 1 : C::BS];
    uint64_t full[C::NSTAGE];
    uint64_t empty[C::NSTAGE];
    uint64_t qfull[C::NQ];
    uint64_t qempty[C::NQ];
    uint64_t xfree;                // the leaders of a unit are done with the state slots
    UnitDesc unit[C::NQ];
    uint32_t issued[C::NSTAGE];    // tiles issued into each stage (producer)
    uint32_t consumed[C::NSTAGE];  // tiles consumed from each stage (consumers)
    uint32_t qissued[C::NQ];
    uint32_t qconsumed[C::NQ];
    volatile int32_t abort;
};

// Byte offset of 16-byte chunk c16 of row t inside a swizzled tile.  The tile is stored
// as [D/64][BS][128 B], each 128-byte line with its 16-byte chunks permuted by
// (line index % 8): the TMA 128B swizzle.
template <class C>
__device__ __forceinline__ uint32_t swz(int t, int c16) {
    return (uint32_t)((c16 >> 3) * C::HALF_BYTES + t * 128 + ((((c16 & 7) ^ (t & 7))) << 4));
}

// ---------------------------------------------------------------------------------
// Output / partial writers shared by both consumer types.
// ---------------------------------------------------------------------------------
// Row of `out` (in rows of head_size) that query row u.row0 + h of a unit goes to.
template <class C>
__device__ __forceinline__ size_t out_row(const DecodeParams& p, const UnitDesc& u, int h) {
    if constexpr (C::kMq) {
        const int r = u.row0 + h, j = r / p.group;
        return ((size_t)u.seq * p.q_len + j) * p.num_q_heads + (size_t)u.kvh * p.group + (r - j * p.group);
    } else {
        return (size_t)u.seq * p.num_q_heads + (size_t)u.kvh * p.group + h;
    }
}

// Row of the partial buffers (part_acc / part_ml) of query row u.row0 + h in slot pslot.
__device__ __forceinline__ size_t part_row(const DecodeParams& p, const UnitDesc& u, int32_t pslot,
                                          int h) {
    return ((size_t)pslot * p.num_kv_heads + u.kvh) * p.rows + u.row0 + h;
}

template <class C>
__device__ __forceinline__ void store_row16(const DecodeParams& p, size_t row, int d0,
                                            const float (&v)[4]) {
    uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + row * C::D + d0;
    uint2 w;
    w.x = pack2<C::kBf16>(v[0], v[1]);
    w.y = pack2<C::kBf16>(v[2], v[3]);
    *reinterpret_cast<uint2*>(o) = w;
}

// The last finished unit of a (sequence, kv head) merges every partition's partial:
//   out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p,
// as one online pass over the partitions, four at a time so that each lane has 4 x NI
// independent L2 loads in flight.  Lane handles (head, 4 dims) chunks lane, lane + 32,
// ...  Partials were written by other CTAs: read them through L2 (ld.global.cg).
template <class C>
__device__ __forceinline__ void merge_partitions(const DecodeParams& p, const UnitDesc& u, int lane) {
    constexpr int CPH = C::D / 4;                         // 4-dim chunks per head
    constexpr int NI = (C::HCAP * CPH + 31) / 32;         // chunks per lane, at most
    const int nr = u.nrows;
    const int np = u.nparts;
    float M[NI], den[NI], a[NI][4];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        M[i] = -INFINITY;
        den[i] = 0.f;
        a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0.f;
    }
    for (int j0 = 0; j0 < np; j0 += 4) {
        float2 ml[4][NI];
        float4 x[4][NI];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int idx = lane + 32 * i;
                const int j = j0 + jj;
                ml[jj][i] = make_float2(-INFINITY, 0.f);
                x[jj][i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < np && idx < nr * CPH) {
                    const size_t row = part_row(p, u, u.pbase + j, idx / CPH);
                    ml[jj][i] = __ldcg(&p.part_ml[row]);
                    x[jj][i] = __ldcg(reinterpret_cast<const float4*>(p.part_acc + row * C::D) + idx % CPH);
                }
            }
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            float Mn = M[i];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) Mn = fmaxf(Mn, ml[jj][i].x);
            const float f = state_weight(M[i], Mn);
            den[i] *= f;
            a[i][0] *= f;
            a[i][1] *= f;
            a[i][2] *= f;
            a[i][3] *= f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const float w = state_weight(ml[jj][i].x, Mn);
                den[i] += w * ml[jj][i].y;
                a[i][0] += w * x[jj][i].x;
                a[i][1] += w * x[jj][i].y;
                a[i][2] += w * x[jj][i].z;
                a[i][3] += w * x[jj][i].w;
            }
            M[i] = Mn;
        }
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int idx = lane + 32 * i;
        if (idx < nr * CPH) {
            const float inv = den[i] > 0.f ? p.out_scale / den[i] : 0.f;
            float v[4] = {a[i][0] * inv, a[i][1] * inv, a[i][2] * inv, a[i][3] * inv};
            store_row16<C>(p, out_row<C>(p, u, idx / CPH), (idx % CPH) * 4, v);
        }
    }
}

// After this unit's partial is stored: count it, and merge if it was the last one.
template <class C>
__device__ __forceinline__ void finish_partition(const DecodeParams& p, const UnitDesc& u, int lane) {
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        const size_t pair = ((size_t)u.seq * p.num_kv_heads + u.kvh) * (p.row_chunks * p.row_groups) +
                            u.row0 / C::HCAP;
        const int t = atomicAdd(&p.arrive[pair], 1);
        last = (t == u.nparts - 1);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
        __threadfence();
        merge_partitions<C>(p, u, lane);
    }
}

// ---------------------------------------------------------------------------------
// Consumer, tensor-core path.
// ---------------------------------------------------------------------------------
template <class C>
struct MmaConsumer {
    static constexpr int D = C::D, BS = C::BS, NT = C::NT, KS = D / 16, MT = BS / 16;
    // The mma operand type: the cache type for 16-bit caches; fp16 for fp8 caches (an
    // E4M3 value converts to fp16 exactly, and the query is converted once per unit).
    static constexpr bool kMmaBf16 = C::kBf16 && !C::kKv8;
    // P enters the PV product as P_hi + P_lo unless the weights are fp16 (fp8 caches) and
    // the output is bf16, where one fp16 term (2^-12) is already far below the output's
    // own resolution.
    static constexpr bool kSplitP = !(C::kKv8 && C::kBf16);
    uint32_t qb[NT][KS][2];
    float m[NT][2], l[NT][2];
    float acc[KS][NT][4];   // O^T fragments: rows = head dims, cols = query heads
    int32_t lim[NT][2];     // multi-query: tokens below lim[nt][j] are visible to this
                            // lane's column nt*8 + 2*(lane%4) + j (causal, and < tok1)

    // fp8 tiles are read with the head dims permuted so that every thread loads 16
    // contiguous bytes (see tile_fp8); the dot product does not care about the order
    // as long as Q uses the same one.  Dim of mma k-step i, lane quad q, element j:
    static __device__ __forceinline__ int k_dim_fp8(int i, int q, int j) {
        return 32 * q + 16 * (i >> 2) + 4 * (i & 3) + j;
    }
    // fp8 tiles: the token of S^T row x (0..15) of a 16-token group.  The K rows are read
    // in this order so that the P fragments pair tokens (4q, 4q+1) and (4q+2, 4q+3): the
    // order in which the transposing 8-bit ldmatrix hands out the V^T fragments.
    static __device__ __forceinline__ int fp8_row_token(int x) {
        return 4 * ((x & 7) >> 1) + (x & 1) + 2 * (x >> 3);
    }
    // Token (within the tile) of S^T row lane/4 + 8 * (r / 2) of m-tile mt.
    static __device__ __forceinline__ int score_token(int mt, int lane, int r) {
        const int x = (lane >> 2) + 8 * (r >> 1);
        return mt * 16 + (C::kKv8 ? fp8_row_token(x) : x);
    }
    // Output head dim of accumulator (m-tile i, lane, register r).
    static __device__ __forceinline__ int out_dim(int i, int lane, int r) {
        return i * 16 + (lane >> 2) + 8 * (r >> 1);
    }

    __device__ __forceinline__ void load_q(const uint8_t* qbuf, int nrows, int lane) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = nt * 8 + (lane >> 2);
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                uint32_t b0 = 0, b1 = 0;
                if (row < nrows) {
                    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qbuf + (size_t)row * D * 2);
                    if constexpr (C::kKv8) {
                        const int d0 = k_dim_fp8(i, lane & 3, 0);
                        float x0, x1, x2, x3;
                        unpack2<C::kBf16>(q32[d0 >> 1], x0, x1);
                        unpack2<C::kBf16>(q32[(d0 >> 1) + 1], x2, x3);
                        b0 = pack2<false>(x0, x1);
                        b1 = pack2<false>(x2, x3);
                    } else {
                        b0 = q32[(16 * i + 2 * (lane & 3)) >> 1];
                        b1 = q32[(16 * i + 8 + 2 * (lane & 3)) >> 1];
                    }
                }
                qb[nt][i][0] = b0;
                qb[nt][i][1] = b1;
            }
        }
    }

    // Multi-query: query token j of a sequence of length L sits at position L - q_len + j
    // and sees the tokens before and at it.
    __device__ __forceinline__ void set_limits(const DecodeParams& p, const UnitDesc& u, int lane) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = u.row0 + nt * 8 + 2 * (lane & 3) + j;
                lim[nt][j] = min(u.tok1, u.len - p.q_len + r / p.group + 1);
            }
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[i][nt][r] = 0.f;
    }

    // One tile of BS tokens starting at token tile0, `valid` (1..BS) of which belong to
    // the unit.
    __device__ __forceinline__ void tile(const uint8_t* kt, const uint8_t* vt, int valid, int tile0,
                                         float scale_log2, int lane, const void*) {
        if constexpr (C::kKv8) tile_fp8(kt, vt, valid, scale_log2, lane);
        else tile16(kt, vt, valid, tile0, scale_log2, lane);
    }

    // Online softmax over the tile's scores sc (S^T fragments, raw dot products) and the
    // hi / lo split of the weights into B fragments of the PV product.
    __device__ __forceinline__ void softmax_tile(float (&sc)[MT][NT][4], int valid, int tile0,
                                                 float scale_log2, int lane,
                                                 uint32_t (&pb)[MT][NT][2], uint32_t (&pl)[MT][NT][2]) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int tk = score_token(mt, lane, r);
                    float v = sc[mt][nt][r] * scale_log2;
                    bool keep;
                    if constexpr (C::kMq) keep = tile0 + tk < lim[nt][r & 1];
                    else keep = tk < valid;
                    v = keep ? v : -INFINITY;
                    sc[mt][nt][r] = v;
                    mx[r & 1] = fmaxf(mx[r & 1], v);
                }
            float alpha[2], mref[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
                const float mn = fmaxf(m[nt][j], mx[j]);
                // A multi-query column may have seen no token yet (all masked so far):
                // exponentiate against 0 then, so that its weights and rescale are 0, not NaN.
                mref[j] = (C::kMq && mn == -INFINITY) ? 0.f : mn;
                alpha[j] = fast_exp2(m[nt][j] - mref[j]);
                m[nt][j] = mn;
            }
            float ps[2] = {0.f, 0.f};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float e = fast_exp2(sc[mt][nt][r] - mref[r & 1]);
                    sc[mt][nt][r] = e;
                    ps[r & 1] += e;
                }
                const uint32_t h01 = pack2<kMmaBf16>(sc[mt][nt][0], sc[mt][nt][1]);
                const uint32_t h23 = pack2<kMmaBf16>(sc[mt][nt][2], sc[mt][nt][3]);
                float r0, r1, r2, r3;
                unpack2<kMmaBf16>(h01, r0, r1);
                unpack2<kMmaBf16>(h23, r2, r3);
                pb[mt][nt][0] = movmatrix_trans(h01);
                pb[mt][nt][1] = movmatrix_trans(h23);
                if constexpr (kSplitP) {
                    pl[mt][nt][0] = movmatrix_trans(pack2<kMmaBf16>(sc[mt][nt][0] - r0, sc[mt][nt][1] - r1));
                    pl[mt][nt][1] = movmatrix_trans(pack2<kMmaBf16>(sc[mt][nt][2] - r2, sc[mt][nt][3] - r3));
                } else {
                    pl[mt][nt][0] = pl[mt][nt][1] = 0u;
                    (void)r0; (void)r1; (void)r2; (void)r3;
                }
            }
            l[nt][0] = l[nt][0] * alpha[0] + ps[0];
            l[nt][1] = l[nt][1] * alpha[1] + ps[1];
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                acc[i][nt][0] *= alpha[0];
                acc[i][nt][1] *= alpha[1];
                acc[i][nt][2] *= alpha[0];
                acc[i][nt][3] *= alpha[1];
            }
        }
    }

    // fp8 E4M3 tile [BS][128 B] (swizzled).  K: lane (g = lane/4, q = lane%4) reads 16
    // contiguous bytes (k-steps 4h..4h+3 in the permuted head-dim order) of S^T rows g
    // and g+8 of each 16-token group, i.e. of tokens fp8_row_token(g), fp8_row_token(g+8)
    // -- an even and an odd token, whose chunks the 128B swizzle puts in different banks.
    // V^T: the transposing 8-bit ldmatrix gives the lane head dims g and g+8 of tokens
    // 4q .. 4q+3, which widen to fp16 fragments as they stand (k-slots 2q, 2q+1 = tokens
    // 4q, 4q+1; k-slots 2q+8, 2q+9 = tokens 4q+2, 4q+3, matching the P fragments).
    __device__ __forceinline__ void tile_fp8(const uint8_t* kt, const uint8_t* vt, int valid,
                                             float scale_log2, int lane) {
        const int g = lane >> 2, q = lane & 3;
        float sc[MT][NT][4], sc2[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[mt][nt][r] = sc2[mt][nt][r] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int t0 = mt * 16 + fp8_row_token(g), t1 = mt * 16 + fp8_row_token(g + 8);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 w0 = *reinterpret_cast<const uint4*>(kt + swz<C>(t0, 2 * q + h));
                const uint4 w1 = *reinterpret_cast<const uint4*>(kt + swz<C>(t1, 2 * q + h));
                const uint32_t u0[4] = {w0.x, w0.y, w0.z, w0.w};
                const uint32_t u1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int i = 4 * h + s4;
                    uint32_t a[4];
                    e4m3x4_to_f16x2x2(u0[s4], a[0], a[2]);   // row g:   k 2q,2q+1 | 2q+8,2q+9
                    e4m3x4_to_f16x2x2(u1[s4], a[1], a[3]);   // row g+8
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (i & 1) mma_16816<false>(sc2[mt][nt], a, qb[nt][i][0], qb[nt][i][1]);
                        else mma_16816<false>(sc[mt][nt], a, qb[nt][i][0], qb[nt][i][1]);
                    }
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[mt][nt][r] += sc2[mt][nt][r];
        uint32_t pb[MT][NT][2], pl[MT][NT][2];
        softmax_tile(sc, valid, 0, scale_log2, lane, pb, pl);
        const bool ragged = valid < BS;
        const uint32_t vbase = smem_u32(vt);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            // this lane's V^T fragments hold tokens 4q .. 4q+3 of the 16-token group
            uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
            if (ragged) {
                // Rows past the context may hold anything (NaN included): zero them so
                // that 0 * NaN never reaches the accumulator.
                const int tq = mt * 16 + 4 * q;
                keep_lo = ((tq < valid) ? 0x0000ffffu : 0u) | ((tq + 1 < valid) ? 0xffff0000u : 0u);
                keep_hi = ((tq + 2 < valid) ? 0x0000ffffu : 0u) | ((tq + 3 < valid) ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int c2 = 0; c2 < D / 32; ++c2) {
                // head dims 32 c2 .. 32 c2 + 31: two 16x16 byte blocks (tokens x dims)
                uint32_t r[4];
                ldmatrix_b8_trans_x2(r, vbase + swz<C>(mt * 16 + (lane & 15), 2 * c2 + (lane >> 4)));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t a[4];
                    e4m3x4_to_f16x2x2(r[2 * h], a[0], a[2]);       // dim g:   tokens 4q..4q+3
                    e4m3x4_to_f16x2x2(r[2 * h + 1], a[1], a[3]);   // dim g+8
                    if (ragged) {
                        a[0] &= keep_lo;
                        a[1] &= keep_lo;
                        a[2] &= keep_hi;
                        a[3] &= keep_hi;
                    }
                    const int i = 2 * c2 + h;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_16816<false>(acc[i][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
                        if constexpr (kSplitP)
                            mma_16816<false>(acc[i][nt], a, pl[mt][nt][0], pl[mt][nt][1]);
                    }
                }
            }
        }
    }

    __device__ __forceinline__ void tile16(const uint8_t* kt, const uint8_t* vt, int valid,
                                           int tile0, float scale_log2, int lane) {
        const int r8 = lane & 7, mi = lane >> 3;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
        // S^T[token][head] = K Q^T, the head-dim steps split over two accumulator chains
        // (even and odd steps) so that consecutive mma.sync do not wait on each other
        float sc[MT][NT][4], sc2[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[mt][nt][r] = sc2[mt][nt][r] = 0.f;
#pragma unroll
        for (int i = 0; i < KS; ++i) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                const int t = mt * 16 + r8 + 8 * (mi & 1);
                ldmatrix_x4(a, kbase + swz<C>(t, 2 * i + (mi >> 1)));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (i & 1) mma_16816<C::kBf16>(sc2[mt][nt], a, qb[nt][i][0], qb[nt][i][1]);
                    else mma_16816<C::kBf16>(sc[mt][nt], a, qb[nt][i][0], qb[nt][i][1]);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[mt][nt][r] += sc2[mt][nt][r];
        // online softmax; the weights enter the PV product as two 16-bit terms, P = P_hi +
        // P_lo, so that their rounding to the operand type costs ~2^-17 instead of 2^-9
        // (bf16) of relative error.
        uint32_t pb[MT][NT][2], pl[MT][NT][2];
        softmax_tile(sc, valid, tile0, scale_log2, lane, pb, pl);
        // O^T[dim][head] += V^T P^T
        const bool ragged = valid < BS;
#pragma unroll
        for (int i = 0; i < KS; ++i) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                const int t = mt * 16 + r8 + 8 * (mi >> 1);
                ldmatrix_x4_trans(a, vbase + swz<C>(t, 2 * i + (mi & 1)));
                if (ragged) {
                    // Rows past the context may hold anything (NaN included): zero them
                    // so that 0 * NaN never reaches the accumulator.
                    const int t0 = mt * 16 + 2 * (lane & 3);
                    const uint32_t lo0 = (t0 < valid) ? 0x0000ffffu : 0u;
                    const uint32_t hi0 = (t0 + 1 < valid) ? 0xffff0000u : 0u;
                    const uint32_t lo8 = (t0 + 8 < valid) ? 0x0000ffffu : 0u;
                    const uint32_t hi8 = (t0 + 9 < valid) ? 0xffff0000u : 0u;
                    a[0] &= lo0 | hi0;
                    a[1] &= lo0 | hi0;
                    a[2] &= lo8 | hi8;
                    a[3] &= lo8 | hi8;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_16816<C::kBf16>(acc[i][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
                    mma_16816<C::kBf16>(acc[i][nt], a, pl[mt][nt][0], pl[mt][nt][1]);
                }
            }
        }
    }

    __device__ __forceinline__ void export_state(float* buf, int lane) const {
        int k = 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                buf[(k++) * 32 + lane] = m[nt][j];
                buf[(k++) * 32 + lane] = l[nt][j];
            }
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) buf[(k++) * 32 + lane] = acc[i][nt][r];
    }

    __device__ __forceinline__ void merge_state(const float* buf, int lane) {
        float a[NT][2], b[NT][2];
        int k = 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float mo = buf[(k++) * 32 + lane];
                const float lo = buf[(k++) * 32 + lane];
                const float M = fmaxf(m[nt][j], mo);
                a[nt][j] = state_weight(m[nt][j], M);
                b[nt][j] = state_weight(mo, M);
                m[nt][j] = M;
                l[nt][j] = a[nt][j] * l[nt][j] + b[nt][j] * lo;
            }
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float o = buf[(k++) * 32 + lane];
                    acc[i][nt][r] = a[nt][r & 1] * acc[i][nt][r] + b[nt][r & 1] * o;
                }
    }

    // Writes the unit's result: final rows of `out` (pslot < 0) or a partial.
    __device__ __forceinline__ void finish(float* ostage, const DecodeParams& p, const UnitDesc& u,
                                           int lane) {
        float lt[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v = l[nt][j];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                lt[nt][j] = v;
            }
        const bool final_out = u.pslot < 0;
        // one reciprocal per column (query row) this lane holds, not one per element
        float inv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                inv[nt][j] = !final_out ? 1.f : lt[nt][j] > 0.f ? p.out_scale / lt[nt][j] : 0.f;
        // stage [head][dim] in fp32 so the rows leave as contiguous vectors
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int d = out_dim(i, lane, r);
                    const int h = nt * 8 + 2 * (lane & 3) + (r & 1);
                    ostage[h * D + d] = acc[i][nt][r] * inv[nt][r & 1];
                }
        __syncwarp();
        const int nr = u.nrows;
        if (final_out) {
            // rows of a unit are contiguous in `out` unless they span several query tokens
            uint16_t* out = reinterpret_cast<uint16_t*>(p.out);
            for (int c = lane; c < nr * D / 8; c += 32) {
                const float* src = ostage + c * 8;
                uint4 w;
                w.x = pack2<C::kBf16>(src[0], src[1]);
                w.y = pack2<C::kBf16>(src[2], src[3]);
                w.z = pack2<C::kBf16>(src[4], src[5]);
                w.w = pack2<C::kBf16>(src[6], src[7]);
                const int h = c / (D / 8);
                *reinterpret_cast<uint4*>(out + out_row<C>(p, u, h) * D + (size_t)(c - h * (D / 8)) * 8) = w;
            }
        } else {
            float* dst = p.part_acc + part_row(p, u, u.pslot, 0) * D;
            for (int c = lane; c < nr * D / 4; c += 32)
                *reinterpret_cast<float4*>(dst + (size_t)c * 4) =
                    *reinterpret_cast<const float4*>(ostage + c * 4);
            // (m, l) per row: lanes 0..3 hold columns 2*lane, 2*lane+1 of each n-tile
            if (lane < 4) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int h = nt * 8 + 2 * lane + j;
                        if (h < nr) p.part_ml[part_row(p, u, u.pslot, h)] = make_float2(m[nt][j], lt[nt][j]);
                    }
            }
            finish_partition<C>(p, u, lane);
        }
        __syncwarp();
    }
};

// ---------------------------------------------------------------------------------
// Consumer, CUDA-core path: lane owns head dims [lane*DPL, lane*DPL + DPL).
// ---------------------------------------------------------------------------------
template <class C>
struct CoreConsumer {
    static constexpr int D = C::D, BS = C::BS, G = C::HCAP, DPL = D / 32, NC8 = BS / 8;
    float qf[G][DPL];
    float m[G], l[G];
    float acc[G][DPL];

    __device__ __forceinline__ void load_q(const uint8_t* qbuf, int nrows, int lane) {
        const uint16_t* q16 = reinterpret_cast<const uint16_t*>(qbuf);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < DPL; j += 2) {
                float a = 0.f, b = 0.f;
                if (h < nrows) {
                    const uint32_t w =
                        *reinterpret_cast<const uint32_t*>(q16 + (size_t)h * D + lane * DPL + j);
                    unpack2<C::kBf16>(w, a, b);
                }
                qf[h][j] = a;
                qf[h][j + 1] = b;
            }
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int j = 0; j < DPL; ++j) acc[h][j] = 0.f;
        }
    }

    // Loads this lane's DPL elements of row t of a swizzled tile as fp32.
    __device__ __forceinline__ void load_row(const uint8_t* tile, int t, int lane, float (&x)[DPL]) {
        const int byte = lane * DPL * C::ELEM;    // offset inside the unswizzled row
        const uint8_t* ptr = tile + swz<C>(t, byte >> 4) + (byte & 15);
        if constexpr (C::kKv8) {                  // 4 fp8 E4M3 -> fp16 (exact) -> fp32
            static_assert(DPL == 4, "fp8 rows: head_size 128");
            const uint32_t w = *reinterpret_cast<const uint32_t*>(ptr);
            unpack2<false>(e4m3x2_to_f16x2(w & 0xffffu), x[0], x[1]);
            unpack2<false>(e4m3x2_to_f16x2(w >> 16), x[2], x[3]);
        } else if constexpr (DPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(ptr);
            unpack2<C::kBf16>(w.x, x[0], x[1]);
            unpack2<C::kBf16>(w.y, x[2], x[3]);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(ptr);
            unpack2<C::kBf16>(w, x[0], x[1]);
        }
    }

    __device__ __forceinline__ void tile(const uint8_t* kt, const uint8_t* vt, int valid, int,
                                         float scale_log2, int lane, float (*pbuf)[BS]) {
        // 1. logits: chunk tc of 8 tokens leaves token tc*8 + (lane >> 2) in this lane
        float lg[G][NC8];
        const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
#pragma unroll
        for (int tc = 0; tc < NC8; ++tc) {
            float part[G][8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float k[DPL];
                load_row(kt, tc * 8 + u, lane, k);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float s = 0.f;
#pragma unroll
                    for (int j = 0; j < DPL; ++j) s = fmaf(qf[h][j], k[j], s);
                    part[h][u] = s;
                }
            }
            // transposed butterfly over the 32 lanes (9 shuffles for 8 tokens)
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = b4 ? part[h][i] : part[h][i + 4];
                    const float keep = b4 ? part[h][i + 4] : part[h][i];
                    part[h][i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float send = b3 ? part[h][i] : part[h][i + 2];
                    const float keep = b3 ? part[h][i + 2] : part[h][i];
                    part[h][i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                {
                    const float send = b2 ? part[h][0] : part[h][1];
                    const float keep = b2 ? part[h][1] : part[h][0];
                    part[h][0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                float s = part[h][0];
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                lg[h][tc] = (tc * 8 + (lane >> 2) < valid) ? s * scale_log2 : -INFINITY;
            }
        }
        // 2. online softmax update, once per tile
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mx = lg[h][0];
#pragma unroll
            for (int tc = 1; tc < NC8; ++tc) mx = fmaxf(mx, lg[h][tc]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[h], mx);
            const float alpha = fast_exp2(m[h] - mn);
            m[h] = mn;
            float ps = 0.f;
#pragma unroll
            for (int tc = 0; tc < NC8; ++tc) {
                const float e = fast_exp2(lg[h][tc] - mn);
                ps += e;
                if ((lane & 3) == 0) pbuf[h][tc * 8 + (lane >> 2)] = e;
            }
            l[h] = l[h] * alpha + ps;        // per-lane share; summed over lanes at the end
#pragma unroll
            for (int j = 0; j < DPL; ++j) acc[h][j] *= alpha;
        }
        __syncwarp();
        // 3. P V over the valid rows (rows past the context are never touched)
#pragma unroll
        for (int t = 0; t < BS; ++t) {
            if (t < valid) {
                float v[DPL];
                load_row(vt, t, lane, v);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float w = pbuf[h][t];
#pragma unroll
                    for (int j = 0; j < DPL; ++j) acc[h][j] = fmaf(w, v[j], acc[h][j]);
                }
            }
        }
        __syncwarp();
    }

    __device__ __forceinline__ void export_state(float* buf, int lane) const {
        int k = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            buf[(k++) * 32 + lane] = m[h];
            buf[(k++) * 32 + lane] = l[h];
#pragma unroll
            for (int j = 0; j < DPL; ++j) buf[(k++) * 32 + lane] = acc[h][j];
        }
    }

    __device__ __forceinline__ void merge_state(const float* buf, int lane) {
        int k = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mo = buf[(k++) * 32 + lane];
            const float lo = buf[(k++) * 32 + lane];
            const float M = fmaxf(m[h], mo);
            const float a = state_weight(m[h], M), b = state_weight(mo, M);
            m[h] = M;
            l[h] = a * l[h] + b * lo;
#pragma unroll
            for (int j = 0; j < DPL; ++j) acc[h][j] = a * acc[h][j] + b * buf[(k++) * 32 + lane];
        }
    }

    __device__ __forceinline__ void finish(float*, const DecodeParams& p, const UnitDesc& u,
                                           int lane) {
        const bool final_out = u.pslot < 0;
        const int g = p.group;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            // each token's share sits in 4 lanes (bits 0,1 of the lane id): sum over bits 2..4
            float lt = l[h];
            lt += __shfl_xor_sync(0xffffffffu, lt, 4);
            lt += __shfl_xor_sync(0xffffffffu, lt, 8);
            lt += __shfl_xor_sync(0xffffffffu, lt, 16);
            if (h >= g) continue;
            const size_t row = (size_t)u.kvh * g + h;
            if (final_out) {
                const float inv = lt > 0.f ? p.out_scale / lt : 0.f;
                uint16_t* o = reinterpret_cast<uint16_t*>(p.out) +
                              ((size_t)u.seq * p.num_q_heads + row) * D + lane * DPL;
                if constexpr (DPL == 4) {
                    uint2 w;
                    w.x = pack2<C::kBf16>(acc[h][0] * inv, acc[h][1] * inv);
                    w.y = pack2<C::kBf16>(acc[h][2] * inv, acc[h][3] * inv);
                    *reinterpret_cast<uint2*>(o) = w;
                } else {
                    *reinterpret_cast<uint32_t*>(o) = pack2<C::kBf16>(acc[h][0] * inv, acc[h][1] * inv);
                }
            } else {
                float* dst = p.part_acc + ((size_t)u.pslot * p.num_q_heads + row) * D + lane * DPL;
                if constexpr (DPL == 4) {
                    *reinterpret_cast<float4*>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
                } else {
                    *reinterpret_cast<float2*>(dst) = make_float2(acc[h][0], acc[h][1]);
                }
                if (lane == 0)
                    p.part_ml[(size_t)u.pslot * p.num_q_heads + row] = make_float2(m[h], lt);
            }
        }
        if (!final_out) finish_partition<C>(p, u, lane);
    }
};

// ---------------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MIN_CTAS)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                        const int32_t persistent, const int32_t num_units_v1) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem<C>& sm = *reinterpret_cast<DecodeSmem<C>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Multi-query units with several row groups: every consumer of a row group reads
    // every tile of the unit, so a stage is freed by row_groups arrivals.
    const int32_t row_groups = C::kMq ? p.row_groups : 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], (uint32_t)row_groups);
            sm.issued[i] = 0;
            sm.consumed[i] = 0;
        }
        mbar_init(&sm.xfree, 1);   // the unit's leader (kernels with one row group)
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], C::NCONS);
            sm.qissued[i] = 0;
            sm.qconsumed[i] = 0;
        }
        sm.abort = 0;
        fence_barrier_init();
        prefetch_tensor_map(&kmap);
        prefetch_tensor_map(&vmap);
    }
    __syncthreads();
    // Launched as a programmatic dependent of the plan (V2) or reshape (V1) kernel: the
    // set-up above overlaps the predecessor; nothing it writes is read before this.
    grid_dependency_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t policy = l2_evict_first_policy();
        const int32_t total = persistent ? (int32_t)p.hdr->total_units : num_units_v1;
        // V2: the partition size the plan kernel settled on (fixed or adaptive)
        const int32_t P = persistent ? (int32_t)p.hdr->partition_size : 0;
        const int32_t Hkv = p.num_kv_heads, g = p.group;
        const uint32_t qbytes = (uint32_t)(g * C::D * 2);
        // work units per V2 list entry (per (sequence, kv head) in V1): the kv heads, and
        // for multi-query kernels the chunks of query rows, chunk index fastest so that
        // the chunks sharing a K/V stream are claimed together
        const int32_t RC = C::kMq ? p.row_chunks : 1;
        const int32_t upl = Hkv * RC;
        // Unit w as a descriptor: V1 units are (sequence, kv head) from the grid index;
        // V2 units come from the plan's list entry e (seq, partition, base slot, length).
        auto describe = [&](int32_t w, int4 e, bool done) {
            UnitDesc u;
            u.seq = -1;
            u.kvh = 0;
            u.tok0 = 0;
            u.tok1 = 0;
            u.pslot = -1;
            u.pbase = 0;
            u.nparts = 1;
            u.row0 = 0;
            u.nrows = g;
            u.len = 0;
            u.pad[0] = u.pad[1] = 0;
            if (!done) {
                int32_t wu = w;
                if constexpr (C::kMq) {
                    wu = w / RC;
                    u.row0 = (w - wu * RC) * row_groups * C::HCAP;
                    u.nrows = min(row_groups * C::HCAP, p.rows - u.row0);
                }
                u.kvh = wu % Hkv;
                if (!persistent) {
                    u.seq = wu / Hkv;
                    u.tok1 = clamped_len(p, u.seq, u.kvh == 0 && u.row0 == 0);
                    u.len = u.tok1;
                } else {
                    u.seq = e.x;
                    u.tok0 = e.y * P;
                    u.tok1 = min(u.tok0 + P, e.w);
                    u.nparts = e.w > 0 ? (e.w + P - 1) / P : 1;
                    u.pbase = e.z;
                    u.pslot = u.nparts > 1 ? e.z + e.y : -1;
                    u.len = e.w;
                }
            }
            return u;
        };
        // Loads (all lanes, one entry each) block-table entries b0 .. b0+31 of a unit,
        // replacing entries outside the pool by a row past the tensor map (TMA reads zeros).
        auto load_blocks = [&](const UnitDesc& u, int32_t b0, int32_t n) {
            int32_t phys = p.num_blocks;   // past the unit: a row past the tensor map (zeros)
            if (lane < n) {
                phys = p.block_tables[(size_t)u.seq * p.max_blocks_per_seq + b0 + lane];
                if (phys < 0 || phys >= p.num_blocks) {
                    if (u.kvh == 0) flag_error(p.status, PA_DEVERR_BAD_BLOCK_);
                    phys = p.num_blocks;
                }
            }
            return phys;
        };
        const int4 kNoEntry = make_int4(0, 0, 0, 0);
        // The first unit.  Later units are claimed one ahead: the atomic, the list entry
        // and the first block-table entries of unit k+1 are fetched while unit k's tiles
        // are issued, so that a new unit does not start with three dependent loads.
        // Every CTA starts with the unit of its own index (no claim to wait for); the
        // units after the first gridDim.x are claimed from the counter.
        int32_t claimed = 0;   // lane 0: the unit of the last atomic claim
#ifndef PA_STATIC_FIRST_UNIT
#define PA_STATIC_FIRST_UNIT 1
#endif
        const uint32_t claim_base = PA_STATIC_FIRST_UNIT ? gridDim.x : 0u;
        if (!PA_STATIC_FIRST_UNIT && persistent && lane == 0) claimed = (int32_t)atomicAdd(&p.hdr->counter, 1u);
        int32_t w = (PA_STATIC_FIRST_UNIT || !persistent) ? (int32_t)blockIdx.x : __shfl_sync(0xffffffffu, claimed, 0);
        int4 e = (persistent && w < total) ? p.part_list[w / upl] : kNoEntry;
        int32_t pre_phys = 0;       // prefetched first block-table chunk of unit w
        bool have_pre = false;
        uint32_t stage = 0, ephase = 1;
        for (uint32_t it = 0;; ++it) {
            const bool done = w >= total || warp_sees_abort(sm.abort);
            const UnitDesc u = describe(w, e, done);
            const uint32_t qs = it % C::NQ, qphase = ((it / C::NQ) & 1) ^ 1;
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(&sm.qempty[qs], qphase);
                if (ok) {
                    sm.unit[qs] = u;
                    if (u.seq < 0) {
                        mbar_arrive(&sm.qfull[qs]);
                    } else if constexpr (C::kMq) {
                        // the unit's rows may span query tokens: one row copy each
                        constexpr uint32_t kRowBytes = C::D * 2;
                        mbar_arrive_expect_tx(&sm.qfull[qs], (uint32_t)u.nrows * kRowBytes);
                        for (int h = 0; h < u.nrows; ++h) {
                            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) +
                                                 out_row<C>(p, u, h) * kRowBytes;
                            bulk_load(sm.qbuf[qs] + h * kRowBytes, src, kRowBytes, &sm.qfull[qs]);
                        }
                        sm.qissued[qs] += 1;
                    } else {
                        mbar_arrive_expect_tx(&sm.qfull[qs], qbytes);
                        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) +
                                             ((size_t)u.seq * p.num_q_heads + (size_t)u.kvh * g) * C::D * 2;
                        bulk_load(sm.qbuf[qs], src, qbytes, &sm.qfull[qs]);
                        sm.qissued[qs] += 1;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) {
                    flag_error(p.status, PA_DEVERR_TIMEOUT_);
                    sm.abort = 1;
                }
                break;
            }
            if (u.seq < 0) {
                // Every tile of this CTA is issued.  Once all CTAs are here, the kernels
                // queued after this one (the next call's plan / reshape / decode, each waiting
                // for this kernel before it touches what this one uses) may launch: their
                // launch and the plan's work overlap the last tiles.  (Letting them launch
                // when a CTA starts its last unit measured slower: CTAs of the next decode
                // then became resident on the SMs that freed first, several of the largest
                // units on one SM.)
                if (PA_DECODE_TRIGGER && lane == 0) allow_dependent_launch();
                break;
            }
            // The next unit is claimed once at most kClaimLead of this unit's tiles are left
            // to issue: early enough that its claim, list entry and first block-table
            // entries arrive before they are needed, late enough that a CTA does not sit on
            // a claimed unit that an idle CTA could have taken (which hurts the balance when
            // units are long).  Steps: 0 unclaimed, 1 claimed, 2 entry loaded, 3 blocks loaded.
            constexpr int32_t kClaimLead = PA_CLAIM_LEAD;
            int32_t w_next = total;
            int4 e_next = kNoEntry;
            int32_t next_phys = 0;
            int step = 0;
            auto advance_next = [&]() {
                if (step == 0) {
                    if (persistent && lane == 0)
                        claimed = (int32_t)(claim_base + atomicAdd(&p.hdr->counter, 1u));
                    step = 1;
                } else if (step == 1) {
                    w_next = persistent ? __shfl_sync(0xffffffffu, claimed, 0) : total;
                    e_next = (persistent && w_next < total) ? p.part_list[w_next / upl] : kNoEntry;
                    step = 2;
                } else if (step == 2) {
                    if (w_next < total) {
                        const UnitDesc un = describe(w_next, e_next, false);
                        const int32_t nb0 = un.tok0 / C::PBS, nb1 = (un.tok1 + C::PBS - 1) / C::PBS;
                        next_phys = load_blocks(un, nb0, min(32, nb1 - nb0));
                    }
                    step = 3;
                }
            };
            // The unit's paged blocks nb0 .. nb1-1, TB per tile (the last tile's blocks past
            // nb1 read as zeros), block-table entries 32 at a time.
            const int32_t nb0 = u.tok0 / C::PBS, nb1 = (u.tok1 + C::PBS - 1) / C::PBS;
            const int32_t ntiles = (u.tok1 - u.tok0 + C::BS - 1) / C::BS;
            if (ntiles <= kClaimLead) advance_next();
            for (int32_t jb = nb0; jb < nb0 + ntiles * C::TB && ok; jb += 32) {
                const int32_t n = min(32, nb1 - jb);
                const int32_t phys = (jb == nb0 && have_pre) ? pre_phys : load_blocks(u, jb, n);
                const int32_t tile_base = (jb - nb0) / C::TB;   // first tile of this chunk
                for (int32_t i = 0; i < 32 / C::TB && tile_base + i < ntiles; ++i) {
                    int32_t pb[C::TB];
#pragma unroll
                    for (int bi = 0; bi < C::TB; ++bi) pb[bi] = __shfl_sync(0xffffffffu, phys, i * C::TB + bi);
                    if (lane == 0) {
                        ok = mbar_wait(&sm.empty[stage], ephase);
                        if (ok) {
                            mbar_arrive_expect_tx(&sm.full[stage], 2u * C::TILE_BYTES);
#pragma unroll
                            for (int bi = 0; bi < C::TB; ++bi) {
                                const int32_t y = (pb[bi] * Hkv + u.kvh) * C::PBS;
                                const uint32_t off = bi * C::PBS * 128;
#pragma unroll
                                for (int h = 0; h < C::HALVES; ++h) {
                                    tma_load_2d(sm.kv[stage][0] + h * C::HALF_BYTES + off, &kmap, h * 64, y,
                                                &sm.full[stage], policy);
                                    tma_load_2d(sm.kv[stage][1] + h * C::HALF_BYTES + off, &vmap, h * 64, y,
                                                &sm.full[stage], policy);
                                }
                            }
                            sm.issued[stage] += 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        ephase ^= 1;
                    }
                    if (step > 0 || ntiles - (tile_base + i + 1) <= kClaimLead) advance_next();
                }
            }
            if (!ok) {
                if (lane == 0) {
                    flag_error(p.status, PA_DEVERR_TIMEOUT_);
                    sm.abort = 1;
                }
                break;
            }
            while (step < 3) advance_next();
            w = w_next;
            e = e_next;
            pre_phys = next_phys;
            have_pre = w < total;
        }
    } else {
        // ------------------------------------------------------------ consumers
        using Consumer = typename std::conditional<C::kMma, MmaConsumer<C>, CoreConsumer<C>>::type;
        const int c = warp - 1;
        constexpr int kConsThreads = 32 * C::NCONS;
        // A decision every consumer thread must take the same way (abort or go on).
        auto all_agree = [&](bool v) {
            if constexpr (C::NCONS > 1) return consumers_any(v, kConsThreads);
            else return __any_sync(0xffffffffu, v);
        };
        Consumer cons;
        // Row group of this consumer and its place in the group (ts = 0 .. TS-1): the
        // consumers of a row group share its tiles; ordinary kernels have one row group,
        // so TS = NCONS.
        const int TS = C::kMq ? C::NCONS / row_groups : C::NCONS;
        const int rg = C::kMq ? c / TS : 0;
        const int ts = C::kMq ? c - rg * TS : c;
        // Tiles go round robin over the tiles of all units (tile k to consumer k % TS; as
        // NSTAGE is a multiple of TS, a stage always serves the same consumer), and the
        // consumer of a unit's last tile is its leader: it merges the others' states and
        // writes the result while the others already start on the next unit, whose first
        // tiles are theirs.  Multi-query kernels deal each unit's tiles from consumer 0 of
        // the group, which leads.  One consumer barrier per unit, after
        // its tiles, carries every decision to stop (end of work, a timed-out wait, an
        // abort) to all consumers at once.  A consumer's state slot is free again once
        // the previous unit's leader has merged it, which it signals on the xfree
        // barrier; multi-query kernels, whose leaders stage their output in a state slot,
        // keep a second barrier after the output instead.
        uint32_t gtile = 0;   // tiles of all earlier units
        for (uint32_t it = 0;; ++it) {
            const uint32_t qs = it % C::NQ, qphase = (it / C::NQ) & 1;
            bool stop = !mbar_wait_warp(&sm.qfull[qs], qphase);
            if (stop && lane == 0) {
                flag_error(p.status, PA_DEVERR_TIMEOUT_);
                sm.abort = 1;
            }
            stop = stop || warp_sees_abort(sm.abort);
            UnitDesc u = sm.unit[qs];
            if (stop || u.seq < 0) {
                (void)all_agree(true);   // the unit barrier below, from a consumer that stops
                break;
            }
            if constexpr (C::kMq) {   // this consumer's row group
                u.row0 += rg * C::HCAP;
                u.nrows = min(C::HCAP, p.rows - u.row0);
            }
            const bool has_rows = u.nrows > 0;
            cons.load_q(sm.qbuf[qs] + rg * C::HCAP * C::D * 2, u.nrows, lane);
            if constexpr (C::kMq) cons.set_limits(p, u, lane);
            __syncwarp();
            if (lane == 0) {
                if (c == 0) sm.qconsumed[qs] += 1;
                mbar_arrive(&sm.qempty[qs]);
            }
            cons.reset();
            const int32_t b0 = u.tok0 / C::BS;
            const int32_t ntiles = (u.tok1 + C::BS - 1) / C::BS - b0;
            // (multi-query kernels, whose row-group size is a run-time value, keep consumer 0
            // of the group as leader and start each unit with it)
            const int gmod = C::kMq ? 0 : (int)(gtile % (uint32_t)TS);
            const int lead = C::kMq ? 0 : (gmod + ntiles - 1 + TS) % TS;
            for (int32_t j = (ts - gmod + TS) % TS; j < ntiles; j += TS) {
                const uint32_t k = gtile + (uint32_t)j;
                const uint32_t stage = k % C::NSTAGE, fphase = (k / C::NSTAGE) & 1;
                if (warp_sees_abort(sm.abort)) {
                    stop = true;
                    break;
                }
                if (!mbar_wait_warp(&sm.full[stage], fphase)) {
                    if (lane == 0) {
                        flag_error(p.status, PA_DEVERR_TIMEOUT_);
                        sm.abort = 1;
                    }
                    stop = true;
                    break;
                }
                const int tile0 = (b0 + j) * C::BS;
                const int valid = min(C::BS, u.tok1 - tile0);
                // a row group past the last row only keeps the stage accounting
                if (has_rows) {
                    if constexpr (C::kMma)
                        cons.tile(sm.kv[stage][0], sm.kv[stage][1], valid, tile0, p.scale_log2, lane, nullptr);
                    else
                        cons.tile(sm.kv[stage][0], sm.kv[stage][1], valid, tile0, p.scale_log2, lane, sm.pbuf[c]);
                }
                __syncwarp();
                if (lane == 0) {
                    if (rg == 0) sm.consumed[stage] += 1;
                    mbar_arrive(&sm.empty[stage]);
                }
            }
            gtile += (uint32_t)ntiles;
            // the row group's state slots: consumer ts exports to slot (ts - lead - 1) mod TS
            const int xbase = C::kMq ? rg * TS : 0;
            if (TS > 1 && !stop && ts != lead) {
                if (!C::kMq && it > 0 && !mbar_wait_warp(&sm.xfree, (it - 1) & 1)) {
                    if (lane == 0) {
                        flag_error(p.status, PA_DEVERR_TIMEOUT_);
                        sm.abort = 1;
                    }
                    stop = true;
                } else {
                    cons.export_state(sm.xbuf[xbase + (C::kMq ? ts - 1 : (ts - lead - 1 + TS) % TS)], lane);
                }
            }
            if (all_agree(stop)) break;   // the unit barrier (also: the states are in shared memory)
            if (ts == lead) {
                for (int o = 0; o < TS - 1; ++o) cons.merge_state(sm.xbuf[xbase + o], lane);
                if (!C::kMq && TS > 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.xfree);
                }
                // A row group's leader stages its output in the group's first state slot
                // (multi-query), whose state it has just merged, or in its own slot when
                // the group has one consumer.  A slot holds NSTATE * 32 >= HCAP * D floats.
                if (has_rows && !warp_sees_abort(sm.abort))
                    cons.finish(C::kMq ? sm.xbuf[xbase] : sm.ostage, p, u, lane);
            }
            // multi-query: the leaders' staged outputs leave the slots before the next
            // unit's states arrive
            if constexpr (C::kMq) (void)all_agree(false);
        }
    }

    // On a timeout, copies may still be landing in this CTA's shared memory: wait
    // (bounded) for every issued copy that was never consumed before exiting.
    __syncthreads();
    if (threadIdx.x == 0 && sm.abort) {
        for (int i = 0; i < C::NSTAGE; ++i)
            if (sm.issued[i] > sm.consumed[i]) (void)mbar_wait(&sm.full[i], sm.consumed[i] & 1);
        for (int i = 0; i < C::NQ; ++i)
            if (sm.qissued[i] > sm.qconsumed[i]) (void)mbar_wait(&sm.qfull[i], sm.qconsumed[i] & 1);
    }
}

template <class C>
constexpr size_t decode_smem_bytes() {
    return sizeof(DecodeSmem<C>) + 1024;
}

}  // namespace pa
