"""GB300-native verify/accept step of EAGLE-style speculative decoding."""
