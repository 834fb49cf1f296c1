// trace.cu — optional per-phase timing of the library's calls. With
// TPMLP_TRACE=1 in the environment (read once per process), every traced step
// of a call (a kernel launch or a short sequence of them: the first product,
// the partials, the reduce, ...) is bracketed by two CUDA events recorded on
// the caller's stream; tpmlp_trace_read() waits for the recorded events and
// returns one line per step with its name and device time. Steps issued into
// a stream that is being captured into a CUDA graph are not traced. Without
// the variable nothing is recorded and a step costs one branch.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "tpmlp.h"
#include "trace.h"

namespace tpmlp {

namespace {

struct Record {
  const char* phase;
  cudaEvent_t begin, end;
  int device;
};

constexpr size_t kMaxRecords = 1 << 16;  // further steps are counted as dropped

std::mutex g_mu;
std::vector<Record> g_log;
std::vector<Record> g_free;  // event pairs for reuse (phase unused)
long g_dropped = 0;

bool take_pair(int device, cudaEvent_t& a, cudaEvent_t& b) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (size_t i = g_free.size(); i-- > 0;) {
      if (g_free[i].device == device) {
        a = g_free[i].begin;
        b = g_free[i].end;
        g_free.erase(g_free.begin() + static_cast<std::ptrdiff_t>(i));
        return true;
      }
    }
  }
  if (cudaEventCreate(&a) != cudaSuccess) return false;
  if (cudaEventCreate(&b) != cudaSuccess) {
    cudaEventDestroy(a);
    return false;
  }
  return true;
}

}  // namespace

bool trace_enabled() {
  static const bool on = [] {
    const char* e = getenv("TPMLP_TRACE");
    return e && *e && atoi(e) != 0;
  }();
  return on;
}

TraceScope::TraceScope(const char* phase, cudaStream_t s) : phase_(phase), stream_(s) {
  if (!trace_enabled()) return;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess || st != cudaStreamCaptureStatusNone) return;
  if (cudaGetDevice(&device_) != cudaSuccess) return;
  if (!take_pair(device_, begin_, end_)) return;
  if (cudaEventRecord(begin_, s) != cudaSuccess) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_free.push_back(Record{nullptr, begin_, end_, device_});
    return;
  }
  active_ = true;
}

TraceScope::~TraceScope() {
  if (!active_) return;
  const bool ok = cudaEventRecord(end_, stream_) == cudaSuccess;
  std::lock_guard<std::mutex> lk(g_mu);
  if (ok && g_log.size() < kMaxRecords) {
    g_log.push_back(Record{phase_, begin_, end_, device_});
  } else {
    if (ok) ++g_dropped;
    g_free.push_back(Record{nullptr, begin_, end_, device_});
  }
}

}  // namespace tpmlp

using namespace tpmlp;

extern "C" int tpmlp_trace_read(char* buf, size_t bytes, int* records) {
  if (records) *records = 0;
  if (!buf && bytes) return set_error(TPMLP_ERR_ARG, "buf is NULL but bytes = %zu", bytes);
  std::vector<Record> log;
  long dropped = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    log.swap(g_log);
    dropped = g_dropped;
    g_dropped = 0;
  }
  size_t used = 0;
  int written = 0;
  int rc = TPMLP_OK;
  int cur = -1;
  cudaGetDevice(&cur);
  for (const Record& r : log) {
    float ms = -1.f;
    if (cudaSetDevice(r.device) == cudaSuccess && cudaEventSynchronize(r.end) == cudaSuccess)
      cudaEventElapsedTime(&ms, r.begin, r.end);
    char line[96];
    const int len = snprintf(line, sizeof(line), "%s %.6f\n", r.phase, static_cast<double>(ms));
    if (len > 0 && used + static_cast<size_t>(len) < bytes) {
      memcpy(buf + used, line, static_cast<size_t>(len));
      used += static_cast<size_t>(len);
      ++written;
    } else if (rc == TPMLP_OK) {
      rc = set_error(TPMLP_ERR_WORKSPACE, "trace buffer of %zu bytes holds %d of %zu records", bytes, written,
                     log.size());
    }
  }
  if (cur >= 0) cudaSetDevice(cur);
  if (bytes) buf[used] = '\0';
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const Record& r : log) g_free.push_back(Record{nullptr, r.begin, r.end, r.device});
  }
  if (records) *records = written;
  if (rc == TPMLP_OK && dropped > 0)
    rc = set_error(TPMLP_ERR_WORKSPACE, "%ld steps were not recorded (more than %zu since the last read)", dropped,
                   kMaxRecords);
  return rc;
}

extern "C" int tpmlp_trace_enabled(void) { return trace_enabled() ? 1 : 0; }
