// pa_decode.cuh -- the paged decode-attention kernel for sm_103a.
//
// What it computes ("vLLM Project Update" talk, parts on PagedAttention and on the V2
// kernel; "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention" thread, exact
// attention): for each sequence s and query head h,
//     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) v_t,   t < context_len[s],
// where token t lives in row t % block_size of physical block block_tables[s][t / bs],
// kv head h / group.  A work unit is (sequence, kv head, token range): the whole
// context (V1) or one partition of partition_size tokens (V2), whose partial
// (max, exp-sum, unnormalised sum) is merged afterwards by log-sum-exp.
//
// GB300 design (one CTA = 2 warps, several CTAs per SM):
//   * warp 0 (producer) claims work units, copies the unit's query rows with a 1-D bulk
//     copy, and streams the unit's K and V tiles -- one (block, kv head) tile is
//     block_size x head_size contiguous elements -- with 2-D tensor TMA into an
//     NSTAGE-deep ring of shared-memory stages (128-byte swizzle, L2 evict-first).
//   * warp 1 (consumer) runs the online softmax over the tiles as they land:
//       - group >= 2 (GQA): S^T = K_tile Q^T and O^T += V_tile^T P^T on the tensor cores
//         (mma.sync m16n8k16, tokens / head dims on M, the group's query heads on N),
//         P moved from accumulator to operand layout with movmatrix;
//       - group 1 (MHA) or on request: CUDA cores, each lane owning head_size/32 dims,
//         dot products finished by a transposed butterfly reduction.
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

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

struct UnitDesc {
    int32_t seq;     // -1: no more units
    int32_t kvh;
    int32_t tok0;    // first token of the unit (a multiple of block_size)
    int32_t tok1;    // one past the last token
    int32_t pslot;   // partition slot for partial results, -1: write the final output
    int32_t pad[3];
};

template <int D_, int BS_, bool BF16_, bool MMA_, int HCAP_, int NSTAGE_, int NQ_>
struct DecodeCfg {
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr bool kBf16 = BF16_;
    static constexpr bool kMma = MMA_;
    static constexpr int HCAP = HCAP_;             // query heads per unit the kernel holds
    static constexpr int NT = MMA_ ? HCAP_ / 8 : 0;  // mma n-tiles of 8 heads
    static constexpr int NSTAGE = NSTAGE_;
    static constexpr int NQ = NQ_;
    static constexpr int HALVES = D / 64;          // 128-byte swizzle spans 64 elements
    static constexpr int TILE_BYTES = D * BS * 2;  // one (block, kv head) tile of K or V
    static constexpr int HALF_BYTES = BS * 128;
    static constexpr int QROWS = HCAP;
    static constexpr int THREADS = 64;
    static_assert(D == 64 || D == 128, "head_size");
    static_assert(BS == 16 || BS == 32, "block_size");
    static_assert(!MMA_ || HCAP_ == 8 || HCAP_ == 16, "mma heads");
    static_assert(MMA_ || HCAP_ == 1 || HCAP_ == 2 || HCAP_ == 4 || HCAP_ == 8, "heads");
};

template <class C>
struct alignas(1024) DecodeSmem {
    uint8_t kv[C::NSTAGE][2][C::TILE_BYTES];         // stage: K tile then V tile
    alignas(128) uint8_t qbuf[C::NQ][C::QROWS * C::D * 2];
    alignas(128) float ostage[C::QROWS * C::D];      // output staging (consumer)
    float pbuf[C::QROWS][8];                         // CUDA-core path: softmax weights
    uint64_t full[C::NSTAGE];
    uint64_t empty[C::NSTAGE];
    uint64_t qfull[C::NQ];
    uint64_t qempty[C::NQ];
    UnitDesc unit[C::NQ];
    uint32_t issued[C::NSTAGE];    // tiles issued into each stage (producer)
    uint32_t consumed[C::NSTAGE];  // tiles consumed from each stage (consumer)
    uint32_t qissued[C::NQ];
    uint32_t qconsumed[C::NQ];
    volatile int32_t abort;
};

// Byte offset of element pair / chunk inside a swizzled tile: row t, 16-byte chunk c16
// of the head_size-element row.  The tile is stored as [D/64][BS][128 B], each 128-byte
// line with its 16-byte chunks permuted by (line index % 8), the TMA 128B swizzle.
template <class C>
__device__ __forceinline__ uint32_t swz(int t, int c16) {
    return (uint32_t)((c16 >> 3) * C::HALF_BYTES + t * 128 + ((((c16 & 7) ^ (t & 7))) << 4));
}

// ---------------------------------------------------------------------------------
// Consumer, tensor-core path.
// ---------------------------------------------------------------------------------
template <class C>
struct MmaConsumer {
    static constexpr int D = C::D, BS = C::BS, NT = C::NT, KS = D / 16, MT = BS / 16;
    uint32_t qb[NT][KS][2];
    float m[NT][2], l[NT][2];
    float acc[KS][NT][4];   // O^T fragments: rows = head dims, cols = query heads

    __device__ __forceinline__ void load_q(const uint8_t* qbuf, int group, int lane) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = nt * 8 + (lane >> 2);
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                uint32_t b0 = 0, b1 = 0;
                if (row < group) {
                    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qbuf + (size_t)row * D * 2);
                    b0 = q32[(16 * i + 2 * (lane & 3)) >> 1];
                    b1 = q32[(16 * i + 8 + 2 * (lane & 3)) >> 1];
                }
                qb[nt][i][0] = b0;
                qb[nt][i][1] = b1;
            }
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

    // One tile of BS tokens, `valid` (1..BS) of which belong to the unit.
    __device__ __forceinline__ void tile(const uint8_t* kt, const uint8_t* vt, int valid,
                                         float scale_log2, int lane) {
        const int r8 = lane & 7, mi = lane >> 3;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
        // S^T[token][head] = K Q^T
        float sc[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[mt][nt][r] = 0.f;
#pragma unroll
        for (int i = 0; i < KS; ++i) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                const int t = mt * 16 + r8 + 8 * (mi & 1);
                ldmatrix_x4(a, kbase + swz<C>(t, 2 * i + (mi >> 1)));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_16816<C::kBf16>(sc[mt][nt], a, qb[nt][i][0], qb[nt][i][1]);
            }
        }
        // online softmax, per query head (columns 2*(lane&3) and +1 of each n-tile)
        uint32_t pb[MT][NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int tk = mt * 16 + (lane >> 2) + 8 * (r >> 1);
                    float v = sc[mt][nt][r] * scale_log2;
                    v = tk < valid ? v : -INFINITY;
                    sc[mt][nt][r] = v;
                    mx[r & 1] = fmaxf(mx[r & 1], v);
                }
            float alpha[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
                const float mn = fmaxf(m[nt][j], mx[j]);
                alpha[j] = fast_exp2(m[nt][j] - mn);
                m[nt][j] = mn;
            }
            float ps[2] = {0.f, 0.f};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float e = fast_exp2(sc[mt][nt][r] - m[nt][r & 1]);
                    sc[mt][nt][r] = e;
                    ps[r & 1] += e;
                }
                pb[mt][nt][0] = movmatrix_trans(pack2<C::kBf16>(sc[mt][nt][0], sc[mt][nt][1]));
                pb[mt][nt][1] = movmatrix_trans(pack2<C::kBf16>(sc[mt][nt][2], sc[mt][nt][3]));
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
                for (int nt = 0; nt < NT; ++nt)
                    mma_16816<C::kBf16>(acc[i][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
            }
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
        // stage [head][dim] in fp32
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int d = i * 16 + (lane >> 2) + 8 * (r >> 1);
                    const int h = nt * 8 + 2 * (lane & 3) + (r & 1);
                    float v = acc[i][nt][r];
                    if (final_out) {
                        const float den = lt[nt][r & 1];
                        v = den > 0.f ? v / den : 0.f;
                    }
                    ostage[h * D + d] = v;
                }
        __syncwarp();
        write_rows<C>(ostage, p, u, lane, final_out);
        if (!final_out) {
            // (m, l) per head: lanes 0..3 hold heads 2*lane, 2*lane+1 of each n-tile
            if (lane < 4) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int h = nt * 8 + 2 * lane + j;
                        if (h < p.group)
                            p.part_ml[(size_t)u.pslot * p.num_q_heads + u.kvh * p.group + h] =
                                make_float2(m[nt][j], lt[nt][j]);
                    }
            }
        }
        __syncwarp();
    }

    template <class CC>
    static __device__ __forceinline__ void write_rows(const float* ostage, const DecodeParams& p,
                                                      const UnitDesc& u, int lane, bool final_out) {
        const int g = p.group;
        if (final_out) {
            // 16-bit rows, 8 elements (16 bytes) per lane per step
            uint16_t* out = reinterpret_cast<uint16_t*>(p.out) +
                            ((size_t)u.seq * p.num_q_heads + (size_t)u.kvh * g) * CC::D;
            const int chunks = g * CC::D / 8;
            for (int c = lane; c < chunks; c += 32) {
                const float* src = ostage + c * 8;
                uint4 w;
                w.x = pack2<CC::kBf16>(src[0], src[1]);
                w.y = pack2<CC::kBf16>(src[2], src[3]);
                w.z = pack2<CC::kBf16>(src[4], src[5]);
                w.w = pack2<CC::kBf16>(src[6], src[7]);
                *reinterpret_cast<uint4*>(out + (size_t)c * 8) = w;
            }
        } else {
            float* dst = p.part_acc + ((size_t)u.pslot * p.num_q_heads + (size_t)u.kvh * g) * CC::D;
            const int chunks = g * CC::D / 4;
            for (int c = lane; c < chunks; c += 32)
                *reinterpret_cast<float4*>(dst + (size_t)c * 4) =
                    *reinterpret_cast<const float4*>(ostage + c * 4);
        }
    }
};

// ---------------------------------------------------------------------------------
// Consumer, CUDA-core path: lane owns head dims [lane*DPL, lane*DPL + DPL).
// ---------------------------------------------------------------------------------
template <class C>
struct CoreConsumer {
    static constexpr int D = C::D, BS = C::BS, G = C::HCAP, DPL = D / 32;
    float qf[G][DPL];
    float m[G], l[G];
    float acc[G][DPL];
    uint32_t lane_off;   // byte offset of this lane's dims inside a row (before swizzle)

    __device__ __forceinline__ void load_q(const uint8_t* qbuf, int group, int lane) {
        const uint16_t* q16 = reinterpret_cast<const uint16_t*>(qbuf);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < DPL; j += 2) {
                float a = 0.f, b = 0.f;
                if (h < group) {
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
        const int byte = lane * DPL * 2;          // offset inside the unswizzled row
        const int c16 = byte >> 4;
        const uint8_t* ptr = tile + swz<C>(t, c16) + (byte & 15);
        if constexpr (DPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(ptr);
            unpack2<C::kBf16>(w.x, x[0], x[1]);
            unpack2<C::kBf16>(w.y, x[2], x[3]);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(ptr);
            unpack2<C::kBf16>(w, x[0], x[1]);
        }
    }

    __device__ __forceinline__ void tile(const uint8_t* kt, const uint8_t* vt, int valid,
                                         float scale_log2, int lane, float (*pbuf)[8]) {
#pragma unroll
        for (int tc = 0; tc < BS / 8; ++tc) {
            const int nvalid = valid - tc * 8;   // valid tokens in this chunk of 8
            if (nvalid <= 0) break;
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
            // transposed butterfly: afterwards lane holds the full dot product of token
            // (lane >> 2) of the chunk, for every head
            const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
            float logit[G];
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
                logit[h] = ((lane >> 2) < nvalid) ? s * scale_log2 : -INFINITY;
            }
            // online softmax update per head
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mx = logit[h];
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(m[h], mx);
                const float alpha = fast_exp2(m[h] - mn);
                m[h] = mn;
                const float e = fast_exp2(logit[h] - mn);
                l[h] = l[h] * alpha + e;       // per-lane share; summed over tokens at the end
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[h][j] *= alpha;
                if ((lane & 3) == 0) pbuf[h][lane >> 2] = e;
            }
            __syncwarp();
            float pw[G][8];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4 a = *reinterpret_cast<const float4*>(&pbuf[h][0]);
                const float4 b = *reinterpret_cast<const float4*>(&pbuf[h][4]);
                pw[h][0] = a.x; pw[h][1] = a.y; pw[h][2] = a.z; pw[h][3] = a.w;
                pw[h][4] = b.x; pw[h][5] = b.y; pw[h][6] = b.z; pw[h][7] = b.w;
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (u < nvalid) {   // rows past the context are never touched
                    float v[DPL];
                    load_row(vt, tc * 8 + u, lane, v);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int j = 0; j < DPL; ++j) acc[h][j] = fmaf(pw[h][u], v[j], acc[h][j]);
                }
            }
        }
    }

    __device__ __forceinline__ void finish(float* ostage, const DecodeParams& p, const UnitDesc& u,
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
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
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
        (void)ostage;
    }
};

// ---------------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::THREADS)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                        const int32_t persistent, const int32_t num_units_v1) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem<C>& sm = *reinterpret_cast<DecodeSmem<C>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
            sm.issued[i] = 0;
            sm.consumed[i] = 0;
        }
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], 1);
            sm.qissued[i] = 0;
            sm.qconsumed[i] = 0;
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensor_map(&kmap);
            prefetch_tensor_map(&vmap);
        }
        const uint64_t policy = l2_evict_first_policy();
        const int32_t total = persistent ? (int32_t)p.hdr->total_units : num_units_v1;
        const int32_t Hkv = p.num_kv_heads, g = p.group;
        const uint32_t qbytes = (uint32_t)(g * C::D * 2);
        uint32_t stage = 0, ephase = 1;
        bool first = true;
        for (uint32_t it = 0;; ++it) {
            int32_t w;
            if (persistent) {
                int32_t c = 0;
                if (lane == 0) c = (int32_t)atomicAdd(&p.hdr->counter, 1u);
                w = __shfl_sync(0xffffffffu, c, 0);
            } else {
                w = first ? (int32_t)blockIdx.x : total;
            }
            first = false;
            const bool done = w >= total || sm.abort;
            UnitDesc u;
            u.seq = -1;
            u.kvh = 0;
            u.tok0 = 0;
            u.tok1 = 0;
            u.pslot = -1;
            if (!done) {
                u.kvh = w % Hkv;
                if (p.partition_size == 0) {
                    u.seq = w / Hkv;
                    u.tok1 = clamped_len(p, u.seq, u.kvh == 0);
                } else {
                    const int32_t j = w / Hkv;
                    const int2 e = p.part_list[j];
                    u.seq = e.x;
                    const int32_t L = clamped_len(p, u.seq, false);
                    u.tok0 = e.y * p.partition_size;
                    u.tok1 = min(u.tok0 + p.partition_size, L);
                    u.pslot = L > p.partition_size ? j : -1;
                }
            }
            const uint32_t qs = it % C::NQ, qphase = ((it / C::NQ) & 1) ^ 1;
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(&sm.qempty[qs], qphase);
                if (ok) {
                    sm.unit[qs] = u;
                    if (u.seq < 0) {
                        mbar_arrive(&sm.qfull[qs]);
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
            if (u.seq < 0) break;
            const int32_t b0 = u.tok0 / C::BS, b1 = (u.tok1 + C::BS - 1) / C::BS;
            const int32_t* bt_row = p.block_tables + (size_t)u.seq * p.max_blocks_per_seq;
            for (int32_t jb = b0; jb < b1 && ok; jb += 32) {
                const int32_t n = min(32, b1 - jb);
                int32_t phys = 0;
                if (lane < n) {
                    phys = bt_row[jb + lane];
                    if (phys < 0 || phys >= p.num_blocks) {
                        if (u.kvh == 0) flag_error(p.status, PA_DEVERR_BAD_BLOCK_);
                        phys = p.num_blocks;   // past the tensor map's rows: TMA fills zeros
                    }
                }
                for (int32_t i = 0; i < n; ++i) {
                    const int32_t pb = __shfl_sync(0xffffffffu, phys, i);
                    if (lane == 0) {
                        ok = mbar_wait(&sm.empty[stage], ephase);
                        if (ok) {
                            mbar_arrive_expect_tx(&sm.full[stage], 2u * C::TILE_BYTES);
                            const int32_t y = (pb * Hkv + u.kvh) * C::BS;
#pragma unroll
                            for (int h = 0; h < C::HALVES; ++h) {
                                tma_load_2d(sm.kv[stage][0] + h * C::HALF_BYTES, &kmap, h * 64, y,
                                            &sm.full[stage], policy);
                                tma_load_2d(sm.kv[stage][1] + h * C::HALF_BYTES, &vmap, h * 64, y,
                                            &sm.full[stage], policy);
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
                }
            }
            if (!ok) {
                if (lane == 0) {
                    flag_error(p.status, PA_DEVERR_TIMEOUT_);
                    sm.abort = 1;
                }
                break;
            }
        }
    } else {
        // ------------------------------------------------------------ consumer
        using Consumer = typename std::conditional<C::kMma, MmaConsumer<C>, CoreConsumer<C>>::type;
        Consumer cons;
        uint32_t stage = 0, fphase = 0;
        for (uint32_t it = 0;; ++it) {
            const uint32_t qs = it % C::NQ, qphase = (it / C::NQ) & 1;
            if (!mbar_wait(&sm.qfull[qs], qphase)) {
                if (lane == 0) {
                    flag_error(p.status, PA_DEVERR_TIMEOUT_);
                    sm.abort = 1;
                }
                break;
            }
            const UnitDesc u = sm.unit[qs];
            if (u.seq < 0) break;
            cons.load_q(sm.qbuf[qs], p.group, lane);
            __syncwarp();
            if (lane == 0) {
                sm.qconsumed[qs] += 1;
                mbar_arrive(&sm.qempty[qs]);
            }
            cons.reset();
            const int32_t b0 = u.tok0 / C::BS, b1 = (u.tok1 + C::BS - 1) / C::BS;
            bool ok = true;
            for (int32_t b = b0; b < b1; ++b) {
                if (!mbar_wait(&sm.full[stage], fphase)) {
                    ok = false;
                    break;
                }
                const int valid = min(C::BS, u.tok1 - b * C::BS);
                if constexpr (C::kMma) {
                    cons.tile(sm.kv[stage][0], sm.kv[stage][1], valid, p.scale_log2, lane);
                } else {
                    cons.tile(sm.kv[stage][0], sm.kv[stage][1], valid, p.scale_log2, lane, sm.pbuf);
                }
                __syncwarp();
                if (lane == 0) {
                    sm.consumed[stage] += 1;
                    mbar_arrive(&sm.empty[stage]);
                }
                if (++stage == C::NSTAGE) {
                    stage = 0;
                    fphase ^= 1;
                }
            }
            if (!ok) {
                if (lane == 0) {
                    flag_error(p.status, PA_DEVERR_TIMEOUT_);
                    sm.abort = 1;
                }
                break;
            }
            cons.finish(sm.ostage, p, u, lane);
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
