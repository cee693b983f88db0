"""TurboQuant hot path on GB300 (sm_103a): Python binding of the libtq C ABI."""
