// Part of layer.cu's translation unit (included inside its anonymous
// namespace, after the layer's stage loops): CUDA-graph replay of layer calls.

// ---------------------------------------------------------------------------
// CUDA-graph replay of whole layer calls (opt-in, upipe_graphs_enable): the
// launch sequence of a call is captured once on a private stream and replayed
// on the caller's stream by later calls with the same arguments, removing the
// per-launch host gaps that dominate short sequences.
// ---------------------------------------------------------------------------
struct GraphEntry {
  std::vector<unsigned long long> key;
  cudaGraphExec_t exec = nullptr;
  upipe_stats stats{};
};
struct GraphCache {
  std::mutex mu;
  bool on = false;
  std::vector<GraphEntry> entries;  // at most kMaxGraphs; later calls run uncached
  static constexpr size_t kMaxGraphs = 32;
};
GraphCache g_graphs;

cudaStream_t capture_stream() {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

// Runs issue(stream, stats) directly, or through a cached graph of it.
template <typename F>
int run_graphed(std::vector<unsigned long long> key, void* stream, upipe_stats* stats, F&& issue) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool use = false;
  {
    std::lock_guard<std::mutex> g(g_graphs.mu);
    use = g_graphs.on;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (use && (g_prof.on || cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone))
    use = false;  // profiling needs per-launch events; a capturing caller captures the launches itself
  if (!use) return issue(stream, stats);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UPIPE_ECUDA;
  key.push_back(static_cast<unsigned long long>(dev));
  {
    std::lock_guard<std::mutex> g(g_graphs.mu);
    for (const GraphEntry& e : g_graphs.entries)
      if (e.key == key) {
        if (stats) *stats = e.stats;
        return cudaGraphLaunch(e.exec, st) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
      }
    if (g_graphs.entries.size() >= GraphCache::kMaxGraphs) return issue(stream, stats);
  }
  cudaStream_t cap = capture_stream();
  if (!cap || !status_ptr()) return UPIPE_ECUDA;  // lazily created state exists before capture begins
  // Nothing issued on the capture stream executes; the graph launch below
  // orders the work after the caller's prior work on its own stream.
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) != cudaSuccess) return UPIPE_ECUDA;
  upipe_stats local{};
  const int rc = issue(static_cast<void*>(cap), &local);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
  if (rc != UPIPE_OK || ec != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    return rc != UPIPE_OK ? rc : UPIPE_ECUDA;
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) return UPIPE_ECUDA;
  {
    std::lock_guard<std::mutex> g(g_graphs.mu);
    GraphEntry e;
    e.key = std::move(key);
    e.exec = exec;
    e.stats = local;
    g_graphs.entries.push_back(std::move(e));
  }
  if (stats) *stats = local;
  return cudaGraphLaunch(exec, st) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

unsigned long long as_key(const void* p) { return static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(p)); }
