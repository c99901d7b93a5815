// q8_moe.cu -- device-side bucketing of (token, slot) pairs by expert.
//
// The routed-expert step of the ds4 engine (GPU code walkthrough, trace 5;
// MoE C notes, section 1) multiplies each selected expert's weights by the
// rows routed to it, reading only the selected experts.  For a batch of
// tokens the pairs p = t*k + j are grouped per expert so that every touched
// expert's weights are streamed once for all of its rows (the grouped GEMM
// with a per-expert offsets table the pages describe for the packed Metal
// kernels).  Three small kernels, all deterministic:
//   1. k_route_count : one CTA per expert counts its pairs; one more gives
//      out-of-range ids a zero output row and raises Q8_ERANGE (no trap); all
//      of them reset the row maps.
//   2. k_route_plan  : one CTA orders the touched experts by pair count
//      (largest first, ties by id: the big groups start first, which keeps the
//      persistent grid balanced under skewed routing), gives each a size class,
//      a 16-row-aligned range of activation-plane rows and a range of work
//      items of its class.
//   3. k_route_fill  : one CTA per expert lists its pairs in increasing p
//      (block-wide prefix sums), giving the plane-row -> output-row map, the
//      plane-row -> input-row map and the pair -> plane-row map used by the
//      gathering quantiser.
#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {

constexpr int ROUTE_THREADS = 512;

uint64_t route_max_rows(uint64_t n_pairs, uint64_t n_expert) {
    const uint64_t touched = n_pairs < n_expert ? n_pairs : n_expert;
    return n_pairs + 15 * touched + 16;
}

__device__ __forceinline__ int block_sum(int v, int *sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) sh[w] = v;
    __syncthreads();
    int s = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += sh[i];
    return s;
}

// CTA e < n_expert counts expert e's pairs.  CTA n_expert zeroes the output rows
// of pairs whose id is out of range and raises the error word.  Every CTA also
// takes a share of setting the plane-row and pair maps to -1 (padding / no row),
// which the fill kernel then overwrites for the real rows.
__global__ void __launch_bounds__(ROUTE_THREADS) k_route_count(const int32_t *__restrict__ ids, uint64_t n_pairs,
                                                                uint32_t n_expert, int32_t *__restrict__ counts,
                                                                uint32_t out_dim, float *__restrict__ out, int *err,
                                                                int32_t *__restrict__ row_to_out,
                                                                int32_t *__restrict__ src_row, uint64_t max_rows,
                                                                int32_t *__restrict__ dst_row) {
    __shared__ int sh[32];
    const uint64_t nthr = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < max_rows; i += nthr) {
        row_to_out[i] = -1;
        src_row[i] = -1;
    }
    if (dst_row)
        for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_pairs; i += nthr) dst_row[i] = -1;
    const uint32_t e = blockIdx.x;
    if (e == n_expert) {
        // each warp reads 32 consecutive ids; the (rare) bad pairs are zeroed by the whole warp
        const int lane = threadIdx.x & 31;
        const uint64_t nwarp = blockDim.x >> 5;
        for (uint64_t p0 = (uint64_t)(threadIdx.x >> 5) * 32; p0 < n_pairs; p0 += nwarp * 32) {
            const uint64_t p = p0 + lane;
            const int32_t id = p < n_pairs ? __ldg(ids + p) : 0;
            unsigned bad = __ballot_sync(0xffffffffu, p < n_pairs && (id < 0 || (uint32_t)id >= n_expert));
            while (bad) {
                const uint64_t pb = p0 + (uint64_t)(__ffs(bad) - 1);
                bad &= bad - 1u;
                for (uint32_t o = lane; o < out_dim; o += 32) out[pb * out_dim + o] = 0.0f;
                if (lane == 0) raise_error(err, DEV_ERANGE);
            }
        }
        return;
    }
    int cnt = 0;
    for (uint64_t p = threadIdx.x; p < n_pairs; p += blockDim.x) cnt += (__ldg(ids + p) == (int32_t)e);
    cnt = block_sum(cnt, sh);
    if (threadIdx.x == 0) counts[e] = cnt;
}

size_t route_plan_bytes(uint32_t n_expert) {
    return ((sizeof(PlanHeader) + (size_t)n_expert * sizeof(Segment)) + 255) & ~(size_t)255;
}

__device__ __forceinline__ int route_class_tokens(int cls) { return cls == 0 ? 8 : 16; }   // GEMV token group

// Block-wide exclusive scan of (a, b) pairs, one pair per thread; returns the
// totals through *ta / *tb.  sh: 2 * (blockDim.x / 32) ints.
__device__ __forceinline__ void block_scan2(int &a, int &b, int *sh, int *ta, int *tb) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int ia = a, ib = b;   // inclusive within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, ia, o), xb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
        }
    }
    __syncthreads();
    if (lane == 31) {
        sh[w] = ia;
        sh[nw + w] = ib;
    }
    __syncthreads();
    int oa = 0, ob = 0, sa = 0, sb = 0;
    for (int i = 0; i < nw; ++i) {
        if (i < w) {
            oa += sh[i];
            ob += sh[nw + i];
        }
        sa += sh[i];
        sb += sh[nw + i];
    }
    a = oa + ia - a;
    b = ob + ib - b;
    *ta = sa;
    *tb = sb;
}

// One CTA.  Touched experts ordered by count (descending, ties by id); in that
// order the classes are contiguous: [0, n2) tensor-core class, [n2, n_gt8)
// class 1, the rest class 0.  Rows and items are exclusive scans over the order.
// The plan from the experts' pair counts cnt[] (shared memory, read by the whole
// CTA after a barrier); order[] (shared) receives the touched experts by rank and
// row0_of[] each expert's first plane row (-1 untouched).
__device__ void route_plan_core(const int32_t *cnt, int32_t *order, uint32_t n_expert, uint32_t out_dim,
                                uint32_t rows_gemv, uint32_t tc_cap, uint8_t *plans, size_t plan_stride,
                                int32_t *__restrict__ row0_of) {
    __shared__ int tot_sh[3];              // touched, > MOE_TC_MIN_ROWS, > 8
    __shared__ int scan_sh[2 * (ROUTE_THREADS / 32)];
    __shared__ int mark_sh[4];             // item / row scans at the class starts n2 and n_gt8
    if (threadIdx.x < 3) tot_sh[threadIdx.x] = 0;
    for (uint32_t e = threadIdx.x; e < n_expert; e += blockDim.x) row0_of[e] = -1;
    __syncthreads();
    int my_active = 0, my_gt_t = 0, my_gt8 = 0;
    for (uint32_t e = threadIdx.x; e < n_expert; e += blockDim.x) {
        const int ce = cnt[e];
        if (ce > 0) {
            int rank = 0;
            for (uint32_t f = 0; f < n_expert; ++f) {
                const int cf = cnt[f];
                rank += (cf > ce) || (cf == ce && f < e);
            }
            order[rank] = (int32_t)e;   // touched experts take ranks 0..n_active-1
            ++my_active;
            my_gt_t += ce > MOE_TC_MIN_ROWS;
            my_gt8 += ce > 8;
        }
    }
    if (my_active) {
        atomicAdd(&tot_sh[0], my_active);
        atomicAdd(&tot_sh[1], my_gt_t);
        atomicAdd(&tot_sh[2], my_gt8);
    }
    __syncthreads();
    const int n_active = tot_sh[0];
    const int n2 = min(tot_sh[1], (int)tc_cap);
    const int n_gt8 = tot_sh[2];
    const int n_rb_gemv = (int)((out_dim + rows_gemv - 1) / rows_gemv);
    const int m_tiles_tc = (int)((out_dim + 127) / 128);
    auto cls_of = [&](int sp) { return sp < n2 ? 2 : (sp < n_gt8 ? 1 : 0); };
    auto items_of = [&](int sp, int ce) {
        const int k = cls_of(sp);
        if (k == 2) return m_tiles_tc * ((ce + 127) / 128);
        const int tg = route_class_tokens(k);
        return n_rb_gemv * ((ce + tg - 1) / tg);
    };
    // each thread owns a contiguous chunk of sorted positions
    const int chunk = (n_active + (int)blockDim.x - 1) / (int)blockDim.x;
    const int s0 = min(n_active, (int)threadIdx.x * chunk), s1 = min(n_active, s0 + chunk);
    int rows = 0, items = 0;
    for (int sp = s0; sp < s1; ++sp) {
        const int ce = cnt[order[sp]];
        rows += (ce + 15) & ~15;
        items += items_of(sp, ce);
    }
    int rows_total, items_total;
    block_scan2(rows, items, scan_sh, &rows_total, &items_total);
    // scans at the class starts (n2: class 1 starts; n_gt8: class 0 starts)
    if (threadIdx.x < 4) mark_sh[threadIdx.x] = -1;
    __syncthreads();
    {
        int r = rows, it = items;
        for (int sp = s0; sp <= s1; ++sp) {
            if (sp == n2 && sp <= n_active) {
                mark_sh[0] = it;
                mark_sh[1] = r;
            }
            if (sp == n_gt8 && sp <= n_active) {
                mark_sh[2] = it;
                mark_sh[3] = r;
            }
            if (sp == s1) break;
            const int ce = cnt[order[sp]];
            r += (ce + 15) & ~15;
            it += items_of(sp, ce);
        }
    }
    __syncthreads();
    // positions past every chunk (empty trailing classes) take the totals
    const int it_at_n2 = mark_sh[0] >= 0 ? mark_sh[0] : items_total, row_at_n2 = mark_sh[1] >= 0 ? mark_sh[1] : rows_total;
    const int it_at_8 = mark_sh[2] >= 0 ? mark_sh[2] : items_total, row_at_8 = mark_sh[3] >= 0 ? mark_sh[3] : rows_total;
    Segment *segs[ROUTE_CLASSES];
    for (int k = 0; k < ROUTE_CLASSES; ++k)
        segs[k] = reinterpret_cast<Segment *>(reinterpret_cast<PlanHeader *>(plans + k * plan_stride) + 1);
    {
        int r = rows, it = items;
        for (int sp = s0; sp < s1; ++sp) {
            const int e = order[sp], ce = cnt[e];
            const int k = cls_of(sp);
            const int cstart = k == 2 ? 0 : (k == 1 ? n2 : n_gt8);
            const int ibase = k == 2 ? 0 : (k == 1 ? it_at_n2 : it_at_8);
            Segment &sg = segs[k][sp - cstart];
            sg.expert = e;
            sg.row0 = r;
            sg.count = ce;
            sg.item_start = it - ibase;
            row0_of[e] = r;
            r += (ce + 15) & ~15;
            it += items_of(sp, ce);
        }
    }
    if (threadIdx.x == 0) {
        const int nseg[3] = {n_active - n_gt8, n_gt8 - n2, n2};
        const int nitem[3] = {items_total - it_at_8, it_at_8 - it_at_n2, it_at_n2};
        const int rend[3] = {n_active > n_gt8 ? rows_total : 0, n_gt8 > n2 ? row_at_8 : 0, n2 > 0 ? row_at_n2 : 0};
        for (int k = 0; k < ROUTE_CLASSES; ++k) {
            PlanHeader *h = reinterpret_cast<PlanHeader *>(plans + k * plan_stride);
            h->n_segments = nseg[k];
            h->n_items = nitem[k];
            h->n_rows = rows_total;
            h->row_end = rend[k];
        }
    }
}

__global__ void __launch_bounds__(ROUTE_THREADS) k_route_plan(const int32_t *__restrict__ counts, uint32_t n_expert,
                                                               uint32_t out_dim, uint32_t rows_gemv, uint32_t tc_cap,
                                                               uint8_t *plans, size_t plan_stride,
                                                               int32_t *__restrict__ row0_of) {
    extern __shared__ int32_t sh_plan[];   // cnt[n_expert], order[n_expert]
    int32_t *cnt = sh_plan;
    int32_t *order = sh_plan + n_expert;
    for (uint32_t e = threadIdx.x; e < n_expert; e += blockDim.x) cnt[e] = counts[e];
    route_plan_core(cnt, order, n_expert, out_dim, rows_gemv, tc_cap, plans, plan_stride, row0_of);
}

// Small batches (the decode sizes): counting, the plan and the pair lists in one
// CTA, with the ids in shared memory, instead of the three kernels above.  The
// same plan and maps: counts are order-independent, the plan is route_plan_core,
// and warp 0 lists each expert's pairs in increasing p (32 pairs at a time,
// ranks within a batch from the lanes holding the same expert).
constexpr uint32_t ROUTE_SMALL_PAIRS = 2048, ROUTE_SMALL_EXPERTS = 2048;

__global__ void __launch_bounds__(ROUTE_THREADS) k_route_small(const int32_t *__restrict__ ids, uint64_t n_pairs,
                                                                uint32_t k, uint32_t n_expert, int x_per_pair,
                                                                uint32_t out_dim, uint32_t rows_gemv, uint32_t tc_cap,
                                                                uint8_t *plans, size_t plan_stride,
                                                                int32_t *__restrict__ row0_of,
                                                                int32_t *__restrict__ row_to_out,
                                                                int32_t *__restrict__ src_row,
                                                                int32_t *__restrict__ dst_row, uint64_t max_rows,
                                                                float *__restrict__ out, int *err) {
    extern __shared__ int32_t sh_small[];   // ids[n_pairs], cnt[n_expert], order[n_expert], run[n_expert]
    int32_t *ids_s = sh_small;
    int32_t *cnt = ids_s + n_pairs;
    int32_t *order = cnt + n_expert;
    int32_t *run = order + n_expert;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint64_t i = threadIdx.x; i < max_rows; i += blockDim.x) {
        row_to_out[i] = -1;
        src_row[i] = -1;
    }
    if (dst_row)
        for (uint64_t i = threadIdx.x; i < n_pairs; i += blockDim.x) dst_row[i] = -1;
    for (uint32_t e = threadIdx.x; e < n_expert; e += blockDim.x) {
        cnt[e] = 0;
        run[e] = 0;
    }
    for (uint64_t i = threadIdx.x; i < n_pairs; i += blockDim.x) ids_s[i] = __ldg(ids + i);
    __syncthreads();
    // counts; each warp reads 32 consecutive ids and zeroes the (rare) bad pairs' rows
    const uint64_t nwarp = blockDim.x >> 5;
    for (uint64_t p0 = (uint64_t)warp * 32; p0 < n_pairs; p0 += nwarp * 32) {
        const uint64_t p = p0 + lane;
        const int32_t id = p < n_pairs ? ids_s[p] : 0;
        const bool ok = id >= 0 && (uint32_t)id < n_expert;
        if (p < n_pairs && ok) atomicAdd(&cnt[id], 1);
        unsigned bad = __ballot_sync(0xffffffffu, p < n_pairs && !ok);
        while (bad) {
            const uint64_t pb = p0 + (uint64_t)(__ffs(bad) - 1);
            bad &= bad - 1u;
            for (uint32_t o = lane; o < out_dim; o += 32) out[pb * out_dim + o] = 0.0f;
            if (lane == 0) raise_error(err, DEV_ERANGE);
        }
    }
    route_plan_core(cnt, order, n_expert, out_dim, rows_gemv, tc_cap, plans, plan_stride, row0_of);
    __syncthreads();   // row0_of is read back by warp 0
    if (warp == 0) {
        for (uint64_t p0 = 0; p0 < n_pairs; p0 += 32) {
            const uint64_t p = p0 + lane;
            const int32_t id = p < n_pairs ? ids_s[p] : -1;
            const bool ok = id >= 0 && (uint32_t)id < n_expert;
            // lanes holding the same expert; lanes without one get keys of their own
            const unsigned same = __match_any_sync(0xffffffffu, ok ? id : -2 - lane);
            if (ok) {
                const int pos = run[id] + __popc(same & ((1u << lane) - 1u));
                const int row = row0_of[id] + pos;
                row_to_out[row] = (int32_t)p;
                src_row[row] = (int32_t)(x_per_pair ? p : p / k);
                if (dst_row) dst_row[p] = row;
            }
            __syncwarp();
            if (ok && lane == __ffs(same) - 1) run[id] += __popc(same);
            __syncwarp();
        }
    }
}

__global__ void __launch_bounds__(ROUTE_THREADS) k_route_fill(const int32_t *__restrict__ ids, uint64_t n_pairs,
                                                               uint32_t k, int x_per_pair,
                                                               const int32_t *__restrict__ row0_of,
                                                               int32_t *__restrict__ row_to_out,
                                                               int32_t *__restrict__ src_row,
                                                               int32_t *__restrict__ dst_row) {
    __shared__ int warp_tot[ROUTE_THREADS / 32];
    const int e = blockIdx.x;
    const int row0 = row0_of[e];
    if (row0 < 0) return;   // untouched expert (uniform across the CTA)
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int base = 0;
    for (uint64_t p0 = 0; p0 < n_pairs; p0 += blockDim.x) {
        const uint64_t p = p0 + threadIdx.x;
        const bool hit = p < n_pairs && __ldg(ids + p) == e;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) warp_tot[w] = __popc(m);
        __syncthreads();
        int before = 0, total = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
            before += (i < w) ? warp_tot[i] : 0;
            total += warp_tot[i];
        }
        if (hit) {
            const int pos = base + before + __popc(m & ((1u << lane) - 1u));
            row_to_out[row0 + pos] = (int32_t)p;
            src_row[row0 + pos] = (int32_t)(x_per_pair ? p : p / k);
            if (dst_row) dst_row[p] = row0 + pos;
        }
        base += total;
        __syncthreads();
    }
}

cudaError_t launch_route(const int32_t *ids, uint64_t n_tok, uint32_t k, uint32_t n_expert, int x_per_pair,
                         uint32_t out_dim, uint32_t rows_gemv, uint32_t tc_cap, int32_t *counts, int32_t *row0_of,
                         uint8_t *plans, int32_t *row_to_out, int32_t *src_row, int32_t *dst_row, uint64_t max_rows,
                         float *out, int *err, int num_sms, cudaStream_t st) {
    const uint64_t n_pairs = n_tok * k;
    cudaError_t e;
    if (n_pairs <= ROUTE_SMALL_PAIRS && n_expert <= ROUTE_SMALL_EXPERTS) {
        const size_t smem = (n_pairs + 3 * (size_t)n_expert) * sizeof(int32_t);   // <= 32 KB
        k_route_small<<<1, ROUTE_THREADS, smem, st>>>(ids, n_pairs, k, n_expert, x_per_pair, out_dim, rows_gemv, tc_cap,
                                                      plans, route_plan_bytes(n_expert), row0_of, row_to_out, src_row,
                                                      dst_row, max_rows, out, err);
        return cudaGetLastError();
    }
    k_route_count<<<n_expert + 1, ROUTE_THREADS, 0, st>>>(ids, n_pairs, n_expert, counts, out_dim, out, err,
                                                          row_to_out, src_row, max_rows, dst_row);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t plan_smem = 2 * (size_t)n_expert * sizeof(int32_t);
    if (plan_smem > 48 * 1024) {
        if ((e = cudaFuncSetAttribute(k_route_plan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan_smem)) !=
            cudaSuccess)
            return e;
    }
    k_route_plan<<<1, ROUTE_THREADS, plan_smem, st>>>(counts, n_expert, out_dim, rows_gemv, tc_cap, plans,
                                                      route_plan_bytes(n_expert), row0_of);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_route_fill<<<n_expert, ROUTE_THREADS, 0, st>>>(ids, n_pairs, k, x_per_pair, row0_of, row_to_out, src_row,
                                                       dst_row);
    return cudaGetLastError();
}

}  // namespace q8
