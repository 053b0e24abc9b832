// The selection key's sigmoid (sigmoid_key, topk_warp.cuh) compiled for the
// host: reads float32 inputs (raw bits, one per line) on stdin and prints the
// bits of sigmoid_key(x), of order_key(x) and of key_float(order_key(x)), one
// triple per line.  Each step of
// the formula is one correctly rounded float32 operation on both processors,
// so the host result is the device result.
#include <cstdio>

#include "simt_emu.h"
#include "topk_warp.cuh"

int main() {
  unsigned bits;
  while (std::scanf("%u", &bits) == 1) {
    const float x = __uint_as_float(bits);
    std::printf("%u %u %u\n", __float_as_uint(moe_route::sigmoid_key(x)), moe_route::order_key(x),
                __float_as_uint(moe_route::key_float(moe_route::order_key(x))));
  }
  return 0;
}
