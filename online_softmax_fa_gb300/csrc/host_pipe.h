// host_pipe.h -- the ordering logic of the host-buffer forward pass
// (fa_fwd_host), written against an abstract set of stream operations so
// that it can be checked without a GPU.
//
// The heads are cut into chunks; chunk c is copied in on the copy-in
// stream, computed on kernel stream c % 2 once its copy-in is done, and
// copied out on the copy-out stream once its kernel is done.  Everything
// starts after the work already queued on the caller's stream, and the
// caller's stream resumes after the last copy-out.
//
// Errors: a call found wrong before anything is queued returns at once.  A
// failure after the first queued operation (a launch or a copy that the
// runtime refuses half-way) still leaves the caller's stream waiting for
// everything already queued on the library's streams, so the caller may
// release its buffers once that stream is synchronised.
//
// `Ops` supplies, each returning 0 on success and a negative status else:
//   record(Event e, Stream s)    record event e on stream s
//   wait(Stream s, Event e)      stream s waits for event e
//   copy_in(int c)               queue chunk c's copies to the device (kIn)
//   launch(int c, Stream s)      queue chunk c's kernel on stream s
//   copy_out(int c)              queue chunk c's copies to the host (kOut)
// Events are named by kind and chunk (Event{kLoaded, c}, ...).
#pragma once

namespace fa {
namespace pipe {

enum Stream { kCaller = 0, kIn = 1, kComp0 = 2, kComp1 = 3, kOut = 4 };
enum EventKind { kStart = 0, kLoaded = 1, kComputed = 2, kDone = 3 };
struct Event {
    EventKind kind;
    int chunk;
};

// Makes the caller's stream wait for everything queued so far on the
// library's streams (best effort: errors here are not reported, the
// original failure is).
template <class Ops>
void fence_caller(Ops &ops) {
    const Stream lib[4] = {kIn, kComp0, kComp1, kOut};
    for (Stream s : lib)
        if (ops.record(Event{kDone, -1}, s) == 0) ops.wait(kCaller, Event{kDone, -1});
}

template <class Ops>
int run(Ops &ops, int chunks) {
    int rc = ops.record(Event{kStart, -1}, kCaller);
    if (rc != 0) return rc;  // nothing queued yet
    bool queued = false;     // an operation that touches the buffers is queued
    const auto fail = [&](int r) {
        if (queued) fence_caller(ops);
        return r;
    };
    const Stream lib[4] = {kIn, kComp0, kComp1, kOut};
    for (Stream s : lib)
        if ((rc = ops.wait(s, Event{kStart, -1})) != 0) return fail(rc);
    for (int c = 0; c < chunks; ++c) {
        const Stream comp = (c & 1) ? kComp1 : kComp0;
        queued = true;  // a copy may be half-queued even when it reports failure
        if ((rc = ops.copy_in(c)) != 0) return fail(rc);
        if ((rc = ops.record(Event{kLoaded, c}, kIn)) != 0) return fail(rc);
        if ((rc = ops.wait(comp, Event{kLoaded, c})) != 0) return fail(rc);
        if ((rc = ops.launch(c, comp)) != 0) return fail(rc);
        if ((rc = ops.record(Event{kComputed, c}, comp)) != 0) return fail(rc);
        if ((rc = ops.wait(kOut, Event{kComputed, c})) != 0) return fail(rc);
        if ((rc = ops.copy_out(c)) != 0) return fail(rc);
    }
    // the copy-out stream has waited for every kernel, in order, and each
    // kernel for its copy-in: the caller's stream resumes after the last
    // copy-out
    if ((rc = ops.record(Event{kDone, -1}, kOut)) != 0) return fail(rc);
    if ((rc = ops.wait(kCaller, Event{kDone, -1})) != 0) return fail(rc);
    return 0;
}

}  // namespace pipe
}  // namespace fa
