// common.cuh -- device helpers of libfnospec: complex arithmetic on float2 and a
// batched radix-2 Stockham FFT in shared memory.
#pragma once

#include <cuda_runtime.h>

namespace fno {

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cscale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }
__device__ __forceinline__ float2 conjf2(float2 a) { return make_float2(a.x, -a.y); }
// (a+bi)(c+di) = (ac-bd) + (ad+bc)i
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// acc += a*b (complex)
__device__ __forceinline__ void cmac(float2& acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, acc.x);
    acc.x = fmaf(-a.y, b.y, acc.x);
    acc.y = fmaf(a.x, b.y, acc.y);
    acc.y = fmaf(a.y, b.x, acc.y);
}

__device__ __forceinline__ int ilog2(int v) { return 31 - __clz(v); }

// Range-checked builds (compiled with -DFNO_DEBUG, the library
// libfnospec_debug.so): every global store of the kernels that take
// FNO_DBG_PARAM is checked against the output ranges of its launch; a store
// outside them is skipped and sets bit 0 (FNO_DEVERR_BOUNDS) of the plan's
// device error word, which fno_get_device_status reports as FNO_ERR_DEVICE.
// Nothing traps or faults.  A kernel passes FNO_DBG_PARAM last in its
// parameter list, calls FNO_DBG_BEGIN() before any role split (it publishes
// the ranges to the CTA through shared memory with one barrier), and guards
// each store with FNO_DBG_OK(address, bytes).  Without FNO_DEBUG the three
// macros vanish and the kernels compile exactly as without them.
#ifdef FNO_DEBUG
struct fno_dbg_ranges {
    const char* lo[2];
    const char* hi[2];
    unsigned* err;
};
__device__ __forceinline__ fno_dbg_ranges& fno_dbg() {
    __shared__ fno_dbg_ranges r;
    return r;
}
__device__ __forceinline__ bool fno_dbg_check(const void* p, size_t bytes) {
    const char* a = static_cast<const char*>(p);
    const fno_dbg_ranges& r = fno_dbg();
    for (int k = 0; k < 2; ++k)
        if (r.lo[k] && a >= r.lo[k] && a + bytes <= r.hi[k]) return true;
    if (r.err) atomicOr(r.err, 1u /* FNO_DEVERR_BOUNDS */);
    return false;
}
#define FNO_DBG_PARAM , fno::fno_dbg_ranges fno_dbg_in
#define FNO_DBG_BEGIN()                                   \
    do {                                                  \
        if (threadIdx.x == 0) fno::fno_dbg() = fno_dbg_in; \
        __syncthreads();                                  \
    } while (0)
#define FNO_DBG_OK(p, bytes) fno::fno_dbg_check((p), (bytes))
#else
#define FNO_DBG_PARAM
#define FNO_DBG_BEGIN() ((void)0)
#define FNO_DBG_OK(p, bytes) true
#endif

// Programmatic dependent launch (PTX griddepcontrol, sm_90+).  Kernels of the
// layer's main path are launched with programmatic stream serialisation
// (launch_pdl in internal.h) and begin with
//   griddep_wait();              // every earlier grid of the stream has completed
//                                // and its writes are visible
//   griddep_launch_dependents(); // the next grid may be scheduled
// so the next kernel's CTAs can take SMs left idle by this kernel's last
// wave.  Because each kernel triggers only after its own wait, when kernel k+1
// starts, kernel k-1 and everything before it have completed: a kernel may read
// inputs that kernel k does not produce before its own griddep_wait().
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Radix-2 Stockham autosort FFT of length L (power of two >= 2) on S sequences
// stored back to back in shared memory (sequence s at a[s*L .. s*L + L)).
// Stage p (p = 1, 2, 4, ..., L/2) reads a, writes b:
//   i in [0, L/2), k = i mod p, u0 = a[i], u1 = a[i + L/2] * w^k with
//   w = e^{-+ i pi / p}, and b[2i - k] = u0 + u1, b[2i - k + p] = u0 - u1;
// the result is in natural order.  tw[j] = e^{+2 pi i j / L} for j in [0, L)
// (the root for stage p and index k is tw[k * L / (2p)], conjugated for the
// forward transform).  The caller must __syncthreads() before the call; the
// function ends with a __syncthreads() and returns the buffer holding the result.
template <bool INVERSE>
__device__ float2* stockham_radix2(float2* a, float2* b, int L, int S,
                                   const float2* __restrict__ tw) {
    const int half = L >> 1;
    const int lhalf = ilog2(half > 0 ? half : 1);
    const int total = S * half;
    for (int p = 1; p < L; p <<= 1) {
        const int tstep = half / p;
        for (int t = threadIdx.x; t < total; t += blockDim.x) {
            const int s = t >> lhalf;
            const int i = t & (half - 1);
            const float2* x = a + (size_t)s * L;
            float2* y = b + (size_t)s * L;
            const int k = i & (p - 1);
            float2 u0 = x[i];
            float2 w = __ldg(&tw[k * tstep]);
            if (!INVERSE) w.y = -w.y;
            float2 u1 = cmul(x[i + half], w);
            const int j = (i << 1) - k;
            y[j] = cadd(u0, u1);
            y[j + p] = csub(u0, u1);
        }
        __syncthreads();
        float2* tmp = a;
        a = b;
        b = tmp;
    }
    return a;
}

}  // namespace fno
