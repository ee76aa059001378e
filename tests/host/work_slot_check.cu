// Host check of the persistent kernels' work decode (work_slot in sm103.cuh):
// for a grid of (items, heads, block) shapes, every work index maps to a
// distinct (item position, head) pair and every pair is reached; inside a
// block the head is the slow index. Prints "ok" or the first failing shape.
#include <cstdio>
#include <vector>

#include "../../context_document_masked_gb300/csrc/sm103.cuh"

int main() {
  const int items[] = {1, 2, 5, 75, 76, 77, 151, 152, 153, 300, 1001, 4199};
  const int heads[] = {1, 2, 3, 4, 8, 16, 32};
  const int blocks[] = {1, 3, 38, 76, 152, 304};
  for (int n : items)
    for (int h : heads)
      for (int b : blocks) {
        std::vector<int> seen((size_t)n * h, 0);
        for (int w = 0; w < n * h; ++w) {
          const fcp::dev::WorkSlot s = fcp::dev::work_slot(w, n, h, b);
          if (s.pos < 0 || s.pos >= n || s.head < 0 || s.head >= h || seen[(size_t)s.pos * h + s.head]++) {
            std::printf("bad n=%d h=%d b=%d w=%d -> (%d, %d)\n", n, h, b, w, s.pos, s.head);
            return 1;
          }
          // Inside a full block, consecutive indices keep the head while the item advances.
          if (w + 1 < n * h && (w + 1) % b != 0 && (w / (b * h)) == ((w + 1) / (b * h)) &&
              (w / (b * h) + 1) * b <= n) {
            const fcp::dev::WorkSlot t = fcp::dev::work_slot(w + 1, n, h, b);
            if (t.head == s.head && t.pos != s.pos + 1) {
              std::printf("order n=%d h=%d b=%d w=%d\n", n, h, b, w);
              return 1;
            }
          }
        }
      }
  std::printf("ok\n");
  return 0;
}
