// host_pipe_check.cpp -- checks the ordering logic of the host-buffer
// forward pass (online_softmax_fa_gb300/csrc/host_pipe.h) without a GPU.
//
// A fake set of stream operations models CUDA's ordering rules: operations
// on one stream run in order, an event recorded on a stream stands for
// everything queued on it so far, and a stream that waits for an event runs
// nothing after the wait before that.  The pipeline runs against the fake
// once without failures and once with a failure injected at each call in
// turn.  Checked:
//   * success: chunk c's kernel runs after its copy-in, its copy-out after
//     its kernel, and the caller's stream resumes after every copy-out;
//   * failure: the call reports the error, and the caller's next operation
//     depends on every operation that was queued (copies of a refused copy
//     call included, since part of it may have been queued).
// Prints "ok" and exits 0, or prints the first violation and exits 1.
//
// Build: g++ -std=c++17 -I <csrc> host_pipe_check.cpp
#include <cstdio>
#include <functional>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "host_pipe.h"

using namespace fa::pipe;

struct Op {
    std::string what;     // "in c", "k c", "out c", or a marker
    std::vector<int> deps;
};

struct Fake {
    std::vector<Op> ops;
    std::map<int, int> last_on_stream;  // stream -> last op id
    std::map<std::pair<int, int>, int> event_op;  // (kind, chunk) -> op id (-1: empty)
    int calls = 0, fail_at = -1;
    std::set<int> data_ops;  // copies and kernels queued

    int add(int stream, const std::string &what, std::vector<int> deps) {
        auto it = last_on_stream.find(stream);
        if (it != last_on_stream.end()) deps.push_back(it->second);
        ops.push_back(Op{what, deps});
        const int id = static_cast<int>(ops.size()) - 1;
        last_on_stream[stream] = id;
        return id;
    }
    bool fail_now() { return calls++ == fail_at; }

    int record(Event e, Stream s) {
        if (fail_now()) return -6;
        auto it = last_on_stream.find(s);
        event_op[{e.kind, e.chunk}] = it == last_on_stream.end() ? -1 : it->second;
        return 0;
    }
    int wait(Stream s, Event e) {
        if (fail_now()) return -6;
        auto it = event_op.find({e.kind, e.chunk});
        if (it == event_op.end()) return -99;  // waiting on an event never recorded
        std::vector<int> deps;
        if (it->second >= 0) deps.push_back(it->second);
        add(s, "wait", deps);
        return 0;
    }
    int copy_in(int c) {
        // a refused copy call may still have queued part of its copies
        const int id = add(kIn, "in " + std::to_string(c), {});
        data_ops.insert(id);
        return fail_now() ? -6 : 0;
    }
    int launch(int c, Stream s) {
        if (fail_now()) return -6;  // a refused launch queues nothing
        data_ops.insert(add(s, "k " + std::to_string(c), {}));
        return 0;
    }
    int copy_out(int c) {
        const int id = add(kOut, "out " + std::to_string(c), {});
        data_ops.insert(id);
        return fail_now() ? -6 : 0;
    }

    std::set<int> ancestors(int id) const {
        std::set<int> seen;
        std::vector<int> todo{id};
        while (!todo.empty()) {
            const int x = todo.back();
            todo.pop_back();
            for (int d : ops[x].deps)
                if (seen.insert(d).second) todo.push_back(d);
        }
        return seen;
    }
    int find(const std::string &what) const {
        for (size_t i = 0; i < ops.size(); ++i)
            if (ops[i].what == what) return static_cast<int>(i);
        return -1;
    }
};

static int fail(const char *msg, int chunks, int at) {
    std::printf("violation (chunks=%d, failure at call %d): %s\n", chunks, at, msg);
    return 1;
}

int main() {
    for (int chunks = 1; chunks <= 9; ++chunks) {
        // success
        Fake ok;
        if (run(ok, chunks) != 0) return fail("success run returned an error", chunks, -1);
        const int total_calls = ok.calls;
        const int end = ok.add(kCaller, "caller next", {});
        const std::set<int> after = ok.ancestors(end);
        for (int c = 0; c < chunks; ++c) {
            const int in = ok.find("in " + std::to_string(c));
            const int k = ok.find("k " + std::to_string(c));
            const int out = ok.find("out " + std::to_string(c));
            if (in < 0 || k < 0 || out < 0) return fail("a chunk operation is missing", chunks, -1);
            if (!ok.ancestors(k).count(in)) return fail("kernel not after its copy-in", chunks, -1);
            if (!ok.ancestors(out).count(k)) return fail("copy-out not after its kernel", chunks, -1);
            if (!after.count(out)) return fail("caller resumes before a copy-out", chunks, -1);
        }
        // a failure at every call in turn
        for (int at = 0; at < total_calls; ++at) {
            Fake f;
            f.fail_at = at;
            if (run(f, chunks) == 0) return fail("failure not reported", chunks, at);
            const int next = f.add(kCaller, "caller next", {});
            const std::set<int> anc = f.ancestors(next);
            for (int id : f.data_ops)
                if (!anc.count(id)) return fail("caller not fenced on a queued operation", chunks, at);
        }
    }
    std::printf("ok\n");
    return 0;
}
