// sv_selftest.cu -- measures, on the device, the fp32 arithmetic that the
// kernels' certified decisions rely on, against fp64:
//   [0] max |G32 - G64| / kG32Err                 (Gumbel of sv_gumbel.cuh)
//   [1] max |ex2(x) / 2^x - 1| / 2^-21            (x in [-126, 64])
//   [2] max |lg2(x) - log2(x)| / (2^-22 max(1, |log2 x|))   (x in [2^-60, 2^8])
//   [3] skip gaps whose fast evaluation (skip_gap) differs from a binary
//       search over the exact thresholds (a count; must be 0), for draws
//       spread uniformly and draws next to every threshold C_g, within the
//       window where the fast path decides near its 2^-9 margin
//   [4] ids whose fp64 G lies outside the table bounds of the top byte of
//       their fine bits (a count; must be 0): the ordinary ids' upper bound,
//       the top ids' upper and lower bounds
// Fine bits are drawn, for ordinary and top ids alike, from regions where the
// formulas are hardest: uniform, w within 2^-28 of 1 (u next to 255/256, or
// 1 - u near 2^-61 for a top id), w below 2^-29, and u around 3/4 (the
// switch between the two evaluations of -log u).
#include "sv_gumbel.cuh"

namespace sv {

// The largest g in 0..256 with M < C_g (C_0 = 2^64: every M), by bisection.
__device__ int skip_gap_bisect(uint64_t M, const uint64_t *C)
{
    int lo = 0, hi = 256;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (M < C[mid])
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__global__ void selftest_kernel(uint64_t seed, long long n, const uint64_t *C, const float *gtab,
                                const float *gtop, unsigned *out)
{
    float r0 = 0.f, r1 = 0.f, r2 = 0.f;
    unsigned bad = 0, badt = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        uint64_t h = splitmix_out(seed ^ (uint64_t)i);
        uint64_t m;
        const bool top = (i >> 2) & 1;
        switch (i & 3) {
        case 0: m = h >> 12; break;
        case 1: m = ((1ull << 52) - 1) - (h >> 40); break;
        case 2: m = h >> 40; break;
        default: m = (3ull << 58) / 255ull / 2ull - (1ull << 23) + (h >> 40); break;
        }
        double g64 = gumbel64(m, top);
        float g32 = gumbel32(m, top);
        const int cb = (int)(m >> 44);
        if (top ? !((double)gtop[kGTab + cb] <= g64 && g64 <= (double)gtop[cb])
                : !(g64 <= (double)gtab[cb]))
            ++badt;
        r0 = fmaxf(r0, (float)(fabs((double)g32 - g64) / (double)kG32Err));
        float x = -126.f + 190.f * (float)((h >> 11) & 0xFFFFF) * 0x1p-20f;
        double e64 = exp2((double)x);
        r1 = fmaxf(r1, (float)(fabs((double)ex2f(x) / e64 - 1.0) / 0x1p-21));
        float y = exp2f(-60.f + 68.f * (float)(h & 0xFFFFF) * 0x1p-20f);
        double l = log2((double)y);
        r2 = fmaxf(r2, (float)(fabs((double)lg2a(y) - l) / (0x1p-22 * fmax(1.0, fabs(l)))));
        // a skip draw: uniform, or within 2^48 (about 4 margins of the fast
        // path) above or below a threshold C_g, g in 1..256
        const uint64_t h2 = splitmix_out(h);
        const int g = 1 + (int)(h2 % 256u);
        const uint64_t off = h2 >> 16;
        uint64_t M = h2;
        if ((i & 3) == 1)
            M = C[g] - 1u - off;
        else if ((i & 3) == 2)
            M = C[g] + off;
        if (skip_gap(M, C) != skip_gap_bisect(M, C))
            ++bad;
    }
    atomicMax(out + 0, __float_as_uint(r0));
    atomicMax(out + 1, __float_as_uint(r1));
    atomicMax(out + 2, __float_as_uint(r2));
    if (bad)
        atomicAdd(out + 3, bad);
    if (badt)
        atomicAdd(out + 4, badt);
}

cudaError_t selftest_run(uint64_t seed, long long n, const uint64_t *skip, const float *gtab,
                         const float *gtop, double *res, cudaStream_t s)
{
    unsigned *d = nullptr;
    cudaError_t e = cudaMallocAsync((void **)&d, 5 * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    cudaMemsetAsync(d, 0, 5 * sizeof(unsigned), s);
    selftest_kernel<<<256, 256, 0, s>>>(seed, n, skip, gtab, gtop, d);
    unsigned h[5] = {0, 0, 0, 0, 0};
    e = cudaMemcpyAsync(h, d, sizeof h, cudaMemcpyDeviceToHost, s);
    cudaFreeAsync(d, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    for (int i = 0; i < 3; ++i) {
        float f;
        memcpy(&f, &h[i], sizeof f);
        res[i] = f;
    }
    res[3] = (double)h[3];
    res[4] = (double)h[4];
    return e;
}

// Waits that run out: warp 0 waits on an mbarrier that nothing arrives at,
// warp 1 waits for a global word that nothing changes (the grid-barrier
// form), each with the bounded-wait primitives the kernels use and at most
// `limit` tries.  Each latches SV_ERR_TIMEOUT in *err when its wait expires
// and returns; nothing else is touched, so the context stays usable.
__global__ void wait_selftest_kernel(int *err, const unsigned *word, uint32_t limit)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int w = threadIdx.x >> 5;
    bool ok = true;
    if (w == 0)
        ok = mbar_wait_n(&bar, 0, limit);  // phase 0 never completes
    else if (w == 1 && threadIdx.x == 32)
        ok = spin_until_change(word, *word, nullptr, limit);
    if (!ok)
        latch(err, SV_ERR_TIMEOUT);
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_arrive(&bar);  // complete the phase before the CTA exits
}

cudaError_t wait_selftest_run(int *err, const unsigned *word, uint32_t limit, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 64, 0, s>>>(err, word, limit);
    return cudaGetLastError();
}

}  // namespace sv
