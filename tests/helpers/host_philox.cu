// Host-side black-box call of the CUDA toolkit's cuRAND Philox4x32-10 block
// function, for the oracle pin tests: an independent library implementation of
// the generator, called (not copied).  The header's function qualifier macro
// is defined first so that its functions compile for the host too.
// stdin: records of 6 uint32 (counter x, y, z, w; key x, y);
// stdout: the 4 output words of each record.
#define QUALIFIERS static __forceinline__ __host__ __device__
#include <curand_philox4x32_x.h>
#include <cstdio>
#include <vector>

int main() {
    std::vector<unsigned int> in;
    unsigned int buf[6 * 1024];
    size_t n;
    while ((n = std::fread(buf, sizeof(unsigned int), 6 * 1024, stdin)) > 0) in.insert(in.end(), buf, buf + n);
    if (in.size() % 6 != 0) return 2;
    std::vector<unsigned int> out;
    out.reserve(in.size() / 6 * 4);
    for (size_t i = 0; i < in.size(); i += 6) {
        const uint4 c = make_uint4(in[i], in[i + 1], in[i + 2], in[i + 3]);
        const uint2 k = make_uint2(in[i + 4], in[i + 5]);
        const uint4 o = curand_Philox4x32_10(c, k);
        out.push_back(o.x);
        out.push_back(o.y);
        out.push_back(o.z);
        out.push_back(o.w);
    }
    std::fwrite(out.data(), sizeof(unsigned int), out.size(), stdout);
    return 0;
}
