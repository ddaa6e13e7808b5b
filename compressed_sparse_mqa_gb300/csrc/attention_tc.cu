// attention_tc.cu -- prefill attention on the 5th-generation tensor cores.
//
// "DS4 (DwarfStar 4)", Architecture (64 query heads share one KV head, 128-token
// window) and Key Techniques, "KV attention compression" (one softmax over the
// raw window and the kept compressed rows): for query i and head h,
//   o_h = sum_j softmax_j(scale * q_h . K_j) V_j
// over the query's own key set (its window rows, then its selected rows).
//
// Because each query has its own key set, the 64 heads of one query are the only
// operand that is shared by all its keys.  The kernel therefore puts the KEYS on
// the 128-row M side of tcgen05.mma and the heads on N = 64:
//   S^T[key][head] = K[key][:] . Q[head][:]       (A = K tile, K-major; B = Q, K-major)
//   O^T[d][head]  += sum_key V[key][d] P^T[key][head]   (A = V tile, MN-major; B = P^T, MN-major)
// so both products run as M = 128 tiles.  Per query (at most 6 key tiles = 768
// keys), S^T of every tile stays in tensor memory (64 columns per tile), the
// softmax runs once over all of them (no online rescaling): per-head max and
// sum across the 128 TMEM lanes use redux.sync on order-preserving integer keys
// and on fixed-point sums, P^T (fp16) goes to shared memory, and O^T
// accumulates in tensor memory.  Key and value rows are gathered with cp.async
// into 128-byte-swizzled tiles (three buffers, shared by the K and V phases).
// CTAs are persistent: one per SM, looping over queries.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"
#include "tcgen05.cuh"

namespace ds4a {
namespace {

constexpr int kH = 64;               // heads (MMA N)
constexpr int kD = 128;              // head dim
constexpr int kTK = 128;             // keys per tile (MMA M)
constexpr int kMaxTiles = 6;         // keys per query <= 768
constexpr int kThreads = 128;
constexpr int kBufs = 3;
constexpr int kTileBytes = kTK * kD * 2;          // 32 KB: [2 atoms][128 rows][128 B]
constexpr int kQBytes = kH * kD * 2;              // 16 KB: [2 atoms][64 rows][128 B]
constexpr int kPBytes = kMaxTiles * kTK * kH * 2; // 96 KB: [768 rows][128 B]
constexpr uint32_t kOCol = kMaxTiles * kH;        // O^T lives at TMEM columns 384 .. 447
constexpr uint32_t kMaxPolls = 1u << 26;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWinTag = 1LL << 62;

struct SmemLayout {
    static constexpr int q = 0;
    static constexpr int tiles = q + kQBytes;
    static constexpr int p = tiles + kBufs * kTileBytes;
    static constexpr int off = p + kPBytes;                          // long long [768]
    static constexpr int red = off + kMaxTiles * kTK * 8;            // uint32 [4][64] x 2
    static constexpr int mh = red + 2 * 4 * kH * 4;                  // float [64] max, [64] 1/sum
    static constexpr int end = mh + 2 * kH * 4;
};
constexpr size_t kSmemBytes = SmemLayout::end + 1024;

struct Args {
    const uint16_t *q;
    const uint16_t *raw_k;
    const uint16_t *raw_v;
    const uint16_t *comp_k;
    const uint16_t *comp_v;
    const int32_t *sel;
    uint16_t *out;
    unsigned int *err;
    long long n_comp;
    long long q_pos0;
    int T;
    int n_prior;
    int window;
    int k_stride;
    int ratio;
    float scale_log2;
};

DS4A_DEVINL void ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

DS4A_DEVINL uint32_t redux_max_u32(uint32_t v) {
    uint32_t r;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;\n" : "=r"(r) : "r"(v));
    return r;
}
DS4A_DEVINL uint32_t redux_add_u32(uint32_t v) {
    uint32_t r;
    asm volatile("redux.sync.add.u32 %0, %1, 0xffffffff;\n" : "=r"(r) : "r"(v));
    return r;
}
DS4A_DEVINL float key_to_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int N>
DS4A_DEVINL void wait_groups(int n) {
    if (n >= 2) cp_async_wait<2>();
    else if (n == 1) cp_async_wait<1>();
    else cp_async_wait<0>();
}

// gather key (or value) rows c*128 .. c*128+127 of the query into a swizzled tile
DS4A_DEVINL void load_tile(unsigned char *tile, const long long *off, int c, const uint16_t *raw,
                           const uint16_t *comp, int tid) {
    for (int i = tid; i < kTK * (kD / 8); i += kThreads) {
        const int r = i >> 4, ch = i & 15;
        unsigned char *dst = tile + (ch >> 3) * (kTK * 128) + tc::sw128_chunk(r, ch & 7);
        const long long o = off[c * kTK + r];
        if (o < 0) *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        else if (o & kWinTag) cp_async16(dst, raw + ((o & ~kWinTag) + ch * 8));
        else cp_async16(dst, comp + (o + ch * 8));
    }
}

__global__ void __launch_bounds__(kThreads, 1) attn_prefill_tc_kernel(Args a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *q_s = smem + SmemLayout::q;
    unsigned char *tile_s = smem + SmemLayout::tiles;
    unsigned char *p_s = smem + SmemLayout::p;
    long long *off = reinterpret_cast<long long *>(smem + SmemLayout::off);
    uint32_t *red_m = reinterpret_cast<uint32_t *>(smem + SmemLayout::red);
    uint32_t *red_l = red_m + 4 * kH;
    float *s_max = reinterpret_cast<float *>(smem + SmemLayout::mh);
    float *s_inv = s_max + kH;
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_bar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        tc::mbar_init(&s_bar, 1);
        tc::mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    constexpr uint32_t kIdescS = tc::idesc_f16_f32(kTK, kH, false, false);
    constexpr uint32_t kIdescO = tc::idesc_f16_f32(kTK, kH, true, true);
    uint32_t phase = 0;
    bool ok = true;
    pdl_wait();
    pdl_trigger();

    for (int i = blockIdx.x; i < a.T; i += gridDim.x) {
        // ---- the query's key list: window rows, then compressed rows ----
        const long long p = a.q_pos0 + i;
        const long long first = p - a.window + 1 > 0 ? p - a.window + 1 : 0;
        const long long raw0 = first - (a.q_pos0 - a.n_prior);
        const int n_w = static_cast<int>(p - first + 1);
        int n_sel = 0;
        if (a.ratio > 0) {
            if (a.sel) n_sel = a.k_stride;
            else {
                const long long nv = (p + 1) / a.ratio;
                n_sel = static_cast<int>(nv < a.n_comp ? nv : a.n_comp);
            }
        }
        const int n_keys = n_w + n_sel;
        const int n_tiles = (n_keys + kTK - 1) / kTK;
        for (int kx = tid; kx < n_tiles * kTK; kx += kThreads) {
            long long o = -1;
            if (kx < n_w) {
                o = kWinTag | ((raw0 + kx) * kD);
            } else if (kx < n_keys) {
                const long long j = a.sel ? static_cast<long long>(__ldg(a.sel + static_cast<size_t>(i) * a.k_stride + (kx - n_w)))
                                          : static_cast<long long>(kx - n_w);
                if (j >= a.n_comp) record_error(a.err, DS4A_ERR_DEVICE_INDEX);
                else if (j >= 0) o = j * kD;
            }
            off[kx] = o;
        }
        __syncthreads();

        // ---- Q (B operand, K-major) and the first key tiles ----
        for (int idx = tid; idx < kH * (kD / 8); idx += kThreads) {
            const int r = idx >> 4, ch = idx & 15;
            cp_async16(q_s + (ch >> 3) * (kH * 128) + tc::sw128_chunk(r, ch & 7),
                       a.q + (static_cast<size_t>(i) * kH + r) * kD + ch * 8);
        }
        const int pre = n_tiles < kBufs ? n_tiles : kBufs;
        for (int c = 0; c < pre; ++c) {
            load_tile(tile_s + c * kTileBytes, off, c, a.raw_k, a.comp_k, tid);
            cp_async_commit();
        }

        // ---- S^T[key][head] for every tile, into TMEM columns c*64 .. ----
        for (int c = 0; c < n_tiles; ++c) {
            wait_groups<0>(min(n_tiles - 1 - c, 2));
            tc::fence_proxy_async();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                const uint32_t t = tc::smem_u32(tile_s + (c % kBufs) * kTileBytes);
                const uint32_t qa = tc::smem_u32(q_s);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint64_t da = tc::desc_sw128(t + (s / 4) * (kTK * 128) + (s % 4) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(qa + (s / 4) * (kH * 128) + (s % 4) * 32, 16, 1024);
                    tc::mma_f16(tmem + c * kH, da, db, kIdescS, s > 0 ? 1u : 0u);
                }
                tc::commit(&s_bar);
            }
            if (!tc::mbar_wait(&s_bar, phase, kMaxPolls)) ok = false;
            phase ^= 1u;
            tc::fence_after_sync();
            if (c + kBufs < n_tiles) {
                load_tile(tile_s + (c % kBufs) * kTileBytes, off, c + kBufs, a.raw_k, a.comp_k, tid);
                cp_async_commit();
            }
        }
        // every buffer is free again: start the value tiles while the softmax runs
        for (int c = 0; c < pre; ++c) {
            load_tile(tile_s + c * kTileBytes, off, c, a.raw_v, a.comp_v, tid);
            cp_async_commit();
        }

        // ---- softmax over the whole key list, per head (TMEM lane = key, column = head) ----
        float acc[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) acc[h] = -INFINITY;
        for (int c = 0; c < n_tiles; ++c) {
            const bool valid = off[c * kTK + warp * 32 + lane] >= 0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                ld_x32(tmem + lane_base + c * kH + half * 32, r);
                tc::wait_ld();
#pragma unroll
                for (int h = 0; h < 32; ++h)
                    if (valid) acc[half * 32 + h] = fmaxf(acc[half * 32 + h], __uint_as_float(r[h]));
            }
        }
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            const uint32_t m = redux_max_u32(float_key(acc[h]));
            if (lane == (h & 31)) red_m[warp * kH + h] = m;
        }
        __syncthreads();
        if (tid < kH) {
            float m = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) m = fmaxf(m, key_to_float(red_m[w * kH + tid]));
            s_max[tid] = m == -INFINITY ? 0.f : m * a.scale_log2;   // scale > 0: max commutes with it
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < kH; ++h) acc[h] = 0.f;
        for (int c = 0; c < n_tiles; ++c) {
            const int key = c * kTK + warp * 32 + lane;
            const bool valid = off[key] >= 0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                ld_x32(tmem + lane_base + c * kH + half * 32, r);
                tc::wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int h = 0; h < 32; h += 2) {
                    const int hh = half * 32 + h;
                    const float p0 = valid ? exp2f(__uint_as_float(r[h]) * a.scale_log2 - s_max[hh]) : 0.f;
                    const float p1 = valid ? exp2f(__uint_as_float(r[h + 1]) * a.scale_log2 - s_max[hh + 1]) : 0.f;
                    acc[hh] += p0;
                    acc[hh + 1] += p1;
                    pk[h / 2] = pack_half2(p0, p1);
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int ch = half * 4 + q4;   // 16-byte chunk = heads ch*8 .. ch*8+7
                    *reinterpret_cast<uint4 *>(p_s + key * 128 + ((ch ^ (key & 7)) << 4)) =
                        make_uint4(pk[q4 * 4], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
                }
            }
        }
        // per-head sums across the 128 lanes, in 2^-22 fixed point (each lane's sum <= 6)
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            const uint32_t s = redux_add_u32(static_cast<uint32_t>(acc[h] * 4194304.f + 0.5f));
            if (lane == (h & 31)) red_l[warp * kH + h] = s;
        }
        __syncthreads();
        if (tid < kH) {
            uint32_t s = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) s += red_l[w * kH + tid];
            s_inv[tid] = 4194304.f / static_cast<float>(s);
        }

        // ---- O^T[d][head] += V^T P^T over the tiles ----
        for (int c = 0; c < n_tiles; ++c) {
            wait_groups<0>(min(n_tiles - 1 - c, 2));
            tc::fence_proxy_async();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                const uint32_t t = tc::smem_u32(tile_s + (c % kBufs) * kTileBytes);
                const uint32_t pb = tc::smem_u32(p_s);
#pragma unroll
                for (int s = 0; s < kTK / 16; ++s) {
                    const uint64_t da = tc::desc_sw128(t + s * 2048, kTK * 128, 1024);
                    const uint64_t db = tc::desc_sw128(pb + (c * kTK + s * 16) * 128, 8192, 1024);
                    tc::mma_f16(tmem + kOCol, da, db, kIdescO, (c > 0 || s > 0) ? 1u : 0u);
                }
                tc::commit(&s_bar);
            }
            if (!tc::mbar_wait(&s_bar, phase, kMaxPolls)) ok = false;
            phase ^= 1u;
            tc::fence_after_sync();
            if (c + kBufs < n_tiles) {
                load_tile(tile_s + (c % kBufs) * kTileBytes, off, c + kBufs, a.raw_v, a.comp_v, tid);
                cp_async_commit();
            }
        }

        // ---- epilogue: TMEM lane = d, column = head ----
        const int d = warp * 32 + lane;
        uint16_t *o = a.out + static_cast<size_t>(i) * kH * kD + d;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            ld_x32(tmem + lane_base + kOCol + half * 32, r);
            tc::wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                const int hh = half * 32 + h;
                o[hh * kD] = f2h(__uint_as_float(r[h]) * s_inv[hh]);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
    }
    if (!ok && tid == 0) record_error(a.err, DS4A_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

bool attn_prefill_tc_ok(int H, int D, long long max_keys) {
    return H == kH && D == kD && max_keys <= kMaxTiles * kTK;
}

cudaError_t launch_attn_prefill_tc(const uint16_t *q, int T, const uint16_t *raw_k, const uint16_t *raw_v,
                                   int n_prior, int window, const uint16_t *comp_k, const uint16_t *comp_v,
                                   long long n_comp, const int32_t *sel, int k_stride, long long q_pos0,
                                   int ratio, float scale, uint16_t *out, const Ctx &c) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    Args a{q, raw_k, raw_v, comp_k, comp_v, sel, out, c.err, n_comp, q_pos0, T, n_prior, window, k_stride,
           ratio, scale * kLog2e};
    const int grid = T < c.num_sms ? T : c.num_sms;
    return launch(attn_prefill_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, c, 1, a);
}

}  // namespace ds4a
