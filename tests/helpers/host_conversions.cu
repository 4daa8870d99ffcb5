// Host-side black-box conversions from the CUDA toolkit's cuda_fp4.h and
// cuda_fp8.h, used by the oracle pin tests as an independent library reference
// for E2M1 and E4M3 round-to-nearest-even with saturation.
// Reads binary float32 values on stdin, writes one byte per value:
//   mode "e2m1": __nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest)
//   mode "e4m3": __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3)
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cstdio>
#include <cstring>
#include <vector>

int main(int argc, char** argv) {
    if (argc < 2) return 2;
    bool e2m1 = std::strcmp(argv[1], "e2m1") == 0;
    std::vector<float> in;
    float buf[4096];
    size_t n;
    while ((n = std::fread(buf, sizeof(float), 4096, stdin)) > 0) in.insert(in.end(), buf, buf + n);
    std::vector<unsigned char> out(in.size());
    for (size_t i = 0; i < in.size(); ++i) {
        if (e2m1) out[i] = (unsigned char)__nv_cvt_float_to_fp4(in[i], __NV_E2M1, cudaRoundNearest);
        else      out[i] = (unsigned char)__nv_cvt_float_to_fp8(in[i], __NV_SATFINITE, __NV_E4M3);
    }
    std::fwrite(out.data(), 1, out.size(), stdout);
    return 0;
}
