// Test helper: converts binary32 values with the host-side conversion routines
// that ship in CUDA's cuda_fp4.h / cuda_fp8.h headers (a library reference for
// the oracle's E2M1 and E4M3 round-to-nearest-even rules).  Reads n float32
// values from stdin, writes n E2M1 codes then n E4M3 (satfinite) bytes.
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cstdio>
#include <vector>

int main()
{
    std::vector<float> v;
    float f;
    while (std::fread(&f, sizeof(float), 1, stdin) == 1) v.push_back(f);
    std::vector<unsigned char> out(2 * v.size());
    for (size_t i = 0; i < v.size(); ++i) {
        out[i] = (unsigned char)__nv_cvt_float_to_fp4(v[i], __NV_E2M1, cudaRoundNearest);
        out[v.size() + i] = (unsigned char)__nv_cvt_float_to_fp8(v[i], __NV_SATFINITE, __NV_E4M3);
    }
    std::fwrite(out.data(), 1, out.size(), stdout);
    return 0;
}
